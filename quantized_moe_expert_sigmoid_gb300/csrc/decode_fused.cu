// Whole MoE layer in one launch for small batches (T <= 8 tokens): router,
// top-k, route plan, dequantising up/gate + SwiGLU, down projection and the
// weighted combine with the shared expert.
//
// Why one launch: at batch 1 the layer reads ~31.9 MB (4 routed experts +
// the shared expert at 6,193,152 B each, plus the 917,504 B router), which
// GB300's HBM3e delivers in under 5 us; a launch boundary costs about 1-2 us,
// so the three dependent steps (route -> up/gate -> down) share one grid.
// (PocketLLM "Xing4.0-29B-A4B: the design record", section 6: the decode
// step there was launch-bound, with the card idle three quarters of the time.)
//
// Grid: one CTA per SM (its shared memory forces 1 CTA/SM).  Each CTA has
// 24 consumer warps and one producer warp:
//   producer  issues 1D bulk (TMA) copies of weight rows into a ring of
//             32 KB shared-memory stages (full/empty mbarriers per stage);
//             before the programmatic-dependent-launch wait it already
//             fetches this CTA's slice of the shared expert's up/gate rows
//             and its router row (weights are immutable); then it polls
//             (bounded) until every router logit has been written (each a
//             tagged 64-bit word), selects the top-k of every token, builds
//             the route plan and issues the routed experts' up/gate rows and
//             this CTA's rows of every W_down.
//   consumers stage x, compute the router logit of expert `blockIdx.x`,
//             quantise x to 16-bit integers per 32-block (power-of-two
//             scale), stream the up/gate items (three groups of 8 warps
//             take alternate items; warp w computes the gate and the up row
//             of output f0 + w % 8, applies SwiGLU and writes h to global
//             memory), wait (bounded) until every CTA has written its h
//             (a grid-wide counter), then own output
//             rows [c*H/G, (c+1)*H/G): every consumer thread keeps fixed
//             (row, 16-weight) units of W_down, accumulates them over all
//             experts (route weight folded into the activation scale) and the
//             rows are reduced once -- one writer per output, no atomics in
//             global memory.
// Dequantisation is in registers: byte-permute lookups of the 4-bit labels
// (device_utils.cuh) and dp2a (16-bit x 8-bit products) into exact int32
// sums per 16 weights, scaled by the weight block's fp16 scale times the
// activation block's scale.
#include <float.h>

#include <algorithm>

#include "device_utils.cuh"
#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kGroupWarps = 8;      // one up/gate item: 8 warps, one output each
constexpr int kItemGroups = 3;      // up/gate items in work at once
constexpr int kConsumerWarps = kGroupWarps * kItemGroups;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kThreads = kConsumers + 32;  // + one producer warp
constexpr int kProducerWarp = kConsumerWarps;
constexpr int kStage = 32768;
constexpr int kMaxStages = 8;
constexpr int kMaxItems = 192;
constexpr int kMaxSlots = kFusedMaxTokens * 9;  // T shared + T*k routed (k <= 8)
constexpr int kMaxEx = kFusedMaxTokens * 8 + 2;
constexpr int kMaxRowsCta = 32;
constexpr int kUnits = 3;  // down-phase (row, 16-weight) units per consumer thread
constexpr uint32_t kPollLimit = 1u << 24;
constexpr uint32_t kSpinLimit = 1u << 21;
constexpr int kBarConsumers = 1;  // named barrier ids (0 is __syncthreads)
constexpr int kBarPlan = 2;       // producer -> consumers: route plan written
constexpr uint64_t kWaitNs = 500000000ull;  // 0.5 s per copy wait before giving up
constexpr uint32_t kLogitTag = 1u;  // high word of a router logit written in this call

// Ring depth of the compile-time Xing4 instances (the launcher checks that
// the shared-memory plan gave this depth): 6 stages up to two tokens, 3 above.
__host__ __device__ constexpr int xing4_stages(int tt) { return tt <= 2 ? 6 : 3; }

struct Params {
  Layer L;
  const void *x;
  int x_bf16, T;
  const float *wr, *bias;
  int64_t bstride;
  const int32_t *ids_in;
  const float *w_in;
  int32_t *ids_out;
  float *w_out;
  void *out;
  int out_bf16;
  int nstage, fpi;
  int wr_rows_smem;  // router rows held in the last ring stage (0: read from global)
  int hq_cap;        // routes whose quantised h fit in shared memory at once
  unsigned *sync;    // [1] h arrivals, [2] exits ([0] unused)
};

struct Item {
  int16_t kind;  // 0: up/gate rows of `count` outputs from f0; 1: W_down rows [f0, f0 + count)
  int16_t a;     // expert slot
  int32_t f0, count;
};

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float load_x(const void *x, int bf16, int64_t i) {
  if (bf16) return __uint_as_float((uint32_t)reinterpret_cast<const uint16_t *>(x)[i] << 16);
  return reinterpret_cast<const float *>(x)[i];
}

// One item's weight rows into a ring stage: gate rows in the stage's first
// half and up rows in its second (kind 0), or W_down rows (kind 1).  A call,
// not inlined: the producer issues from three places, and one copy of the
// code, warm after the first item, is shorter than three cold ones.
__device__ __noinline__ void issue_copy(const Item it, int eid, uint8_t *dst, uint64_t *bar,
                                        const uint8_t *gu, const uint8_t *dn, int64_t gu_eb, int64_t dn_eb,
                                        int64_t rb, int64_t db, int fpi) {
  if (it.kind == 0) {
    const uint8_t *base = gu + (int64_t)eid * gu_eb;
    const int64_t grow = (int64_t)(it.f0 / kGroupRows) * (2 * kGroupRows) + it.f0 % kGroupRows;
    const uint32_t bytes = (uint32_t)(it.count * rb);
    mbar_arrive_expect_tx(bar, 2 * bytes);
    bulk_g2s(dst, base + grow * rb, bytes, bar);
    bulk_g2s(dst + fpi * rb, base + (grow + kGroupRows) * rb, bytes, bar);
  } else {
    const uint8_t *base = dn + (int64_t)eid * dn_eb + (int64_t)it.f0 * db;
    const uint32_t bytes = (uint32_t)(it.count * db);
    mbar_arrive_expect_tx(bar, bytes);
    bulk_g2s(dst, base, bytes, bar);
  }
}

// W_down units of every remaining expert at one token, in one pass (see the
// down phase of decode_fused_kernel): NU live (row, 16-weight) units per
// thread, rows ct / NPD + (kConsumers / NPD) m, position ct % NPD.
template <int NPD, int NU, int TT>
__device__ __forceinline__ void down_units_t1(const Item *its, int n_rem, const uint8_t *ring, const int *ex_rs,
                                              const int8_t (*rid)[kFusedMaxTokens], const int16_t *hq,
                                              const float *shs, int grp_rs, int ct, int i0, int nst,
                                              float (&acc)[kUnits][TT]) {
  constexpr int kFp = NPD * 16, kDb = NPD / 16 * kSBBytes, kRowStep = kConsumers / NPD;
  const int pos = ct & (NPD - 1), b = pos >> 1;
  const int wofs = (b >> 3) * kSBBytes + 16 + (b & 7) * 16 + (pos & 1) * 8;
  const int dofs = (b >> 3) * kSBBytes + (b & 7) * 2;
#pragma unroll 2
  for (int j = 0; j < n_rem; ++j) {
    const Item itj = its[j];
    const int r = rid[itj.a][0];
    if (r < 0) continue;
    const int ho = ex_rs[itj.a] - grp_rs + r;
    const int16_t *hr = hq + ho * kFp + pos * 16;
    const uint4 ha = *reinterpret_cast<const uint4 *>(hr);
    const uint4 hb2 = *reinterpret_cast<const uint4 *>(hr + 8);
    const float sh = shs[ho * (kFp / 32) + b];
    const int stg = nst == 6 ? (i0 + j) % 6 : (i0 + j) % 3;
    const uint8_t *st = ring + (size_t)stg * kStage + (ct / NPD) * kDb;
#pragma unroll
    for (int m = 0; m < NU; ++m) {
      const uint2 q = *reinterpret_cast<const uint2 *>(st + kRowStep * kDb * m + wofs);
      const float d = __half2float(*reinterpret_cast<const __half *>(st + kRowStep * kDb * m + dofs));
      uint32_t c0, c1, c2, c3;
      iq4_decode8(q.x, c0, c1);
      iq4_decode8(q.y, c2, c3);
      const int s0 = dot8_dp2a(c0, c1, ha, 0);
      const int s1 = dot8_dp2a(c2, c3, hb2, 0);
      acc[m][0] = fmaf((float)(s0 + s1), d * sh, acc[m][0]);
    }
  }
}

// NP > 0: rows of Hp = NP * 512 weights (NP 16-weight positions per lane),
// at most 64 experts, bf16 x; NPD > 0: W_down rows of Fp = NPD * 16 weights.
// With both known at compile time every shared-memory offset in the inner
// loops is a per-lane base plus an immediate.  NP = NPD = 0: any shape,
// runtime loops.
template <int TT, int NP, int NPD>
__global__ void __launch_bounds__(kThreads, 1) decode_fused_kernel(const Params p) {
  // router logits held per lane in the top-k: E <= 64 for the compile-time
  // Xing4 shape, up to 256 otherwise.  Code that runs once per call comes
  // from a cold instruction cache, so its length is its cost.
  constexpr int kNloc = NP > 0 ? 2 : 8;
  extern __shared__ __align__(1024) uint8_t smem[];
  __shared__ uint64_t full_bar[kMaxStages], empty_bar[kMaxStages], wr_bar;
  __shared__ Item items[kMaxItems];
  __shared__ int n_items, n_shared_items, n_ex, status, n_issued, last_cta;
  __shared__ int r_tok[kMaxSlots];
  __shared__ float r_w[kMaxSlots];
  __shared__ int ex_id[kMaxEx], ex_rs[kMaxEx + 1];
  __shared__ int8_t rid[kMaxEx][kFusedMaxTokens];  // route of token t inside expert a, or -1
  __shared__ int skey[kFusedMaxTokens * 8], sorted_id[kFusedMaxTokens * 8];
  __shared__ int sel_id[kFusedMaxTokens][8];
  __shared__ float sel_w[kFusedMaxTokens][8];
  __shared__ float red[kConsumerWarps][TT];

  const Layer &L = p.L;
  // the one-token instance is only launched for T = 1
  const int T = TT == 1 ? 1 : p.T, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = gridDim.x, c = blockIdx.x;
  const int Hp = L.Hp, Fp = L.Fp, H = L.H, E = L.E, S = L.S, K = L.k;
  const int64_t rb = L.gu_row_bytes, db = L.dn_row_bytes;
  // divisors known at compile time in the Xing4 instance
  const int nst = NP > 0 ? xing4_stages(TT) : p.nstage, hb = NP > 0 ? NP * 16 : Hp / 32, fb32 = Fp / 32;
  // ring stage and round of item i: the depth is 3 or 6, so both are
  // divisions by a constant (a runtime divisor costs a long sequence)
  auto stage_of = [nst](int i) { return nst == 6 ? i % 6 : i % 3; };
  auto round_of = [nst](int i) { return nst == 6 ? i / 6 : i / 3; };
  uint8_t *ring = smem;
  int16_t *xq = reinterpret_cast<int16_t *>(smem + (size_t)nst * kStage);
  float *sx = reinterpret_cast<float *>(xq + (size_t)T * Hp);
  int16_t *hq = reinterpret_cast<int16_t *>(sx + (size_t)T * hb);
  float *shs = reinterpret_cast<float *>(hq + (size_t)p.hq_cap * Fp);
  // 32-bit splits (H * G, Fp * G and the routed rows * G stay below 2^32;
  // a 64-bit division is a long software sequence)
  const unsigned uG = (unsigned)G;
  const int n0 = (int)((unsigned)c * (unsigned)H / uG), n1 = (int)((unsigned)(c + 1) * (unsigned)H / uG);
  const int nrows = n1 - n0;
  const bool do_route = p.ids_in == nullptr;

  auto add_upgate = [&](int a, int fb, int fe) {  // thread-serial
    int f = fb;
    while (f < fe && n_items < kMaxItems) {
      const int grp_end = (f / kGroupRows + 1) * kGroupRows;
      const int cnt = min(min(fe, grp_end) - f, p.fpi);
      items[n_items++] = Item{0, (int16_t)a, f, cnt};
      f += cnt;
    }
  };

  // ---- set-up ----
  if (tid == 0) {
    for (int s = 0; s < nst; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], kConsumerWarps);
    }
    mbar_init(&wr_bar, 1);
    fence_mbar_init();
    n_items = 0;
    n_ex = 0;
    status = 0;
    ex_rs[0] = 0;
    if (S) {
      ex_id[0] = E;
      ex_rs[1] = T;
      n_ex = 1;
      for (int t = 0; t < T; ++t) {
        r_tok[t] = t;
        r_w[t] = 1.0f;
        rid[0][t] = (int8_t)t;
      }
      add_upgate(0, (int)((unsigned)c * (unsigned)Fp / uG), (int)((unsigned)(c + 1) * (unsigned)Fp / uG));
    }
    n_shared_items = n_items;
  }
  __syncthreads();

  if (warp == kProducerWarp) {
    // =========================== producer warp ===========================
    auto issue = [&](int i) {
      const Item it = items[i];
      const int s = stage_of(i);
      issue_copy(it, ex_id[it.a], ring + (size_t)s * kStage, &full_bar[s], L.gu, L.dn, L.gu_expert_bytes,
                 L.dn_expert_bytes, rb, db, p.fpi);
    };
    int issued = 0;
    if (lane == 0) {
      // the router rows first (the routing is on the critical path), then
      // the shared expert's rows, known before routing
      if (do_route && p.wr_rows_smem > 0) {  // router rows -> last stage (no shared item uses it)
        int nr = 0;
        for (int e = c; e < E; e += G) ++nr;
        if (nr > 0) {
          mbar_arrive_expect_tx(&wr_bar, (uint32_t)(nr * H * 4));
          int r = 0;
          for (int e = c; e < E; e += G, ++r)
            bulk_g2s(ring + (size_t)(nst - 1) * kStage + (size_t)r * H * 4, p.wr + (int64_t)e * H,
                     (uint32_t)(H * 4), &wr_bar);
        }
      }
      // a router CTA lets its router row land first: HBM is busy with every
      // CTA's shared-expert rows at this point, and the routing is what the
      // whole grid waits for
      if (do_route && p.wr_rows_smem > 0 && c < E && !mbar_wait_bounded(&wr_bar, 0, kPollLimit))
        atomicOr(&status, 2);
      for (; issued < n_shared_items && issued < nst; ++issued) issue(issued);
      if (S && nrows > 0)  // the shared expert's W_down rows of this CTA
        bulk_prefetch_l2(L.dn + (int64_t)E * L.dn_expert_bytes + (int64_t)n0 * db, (uint32_t)(nrows * db));
    }
    if (do_route && p.wr_rows_smem == 0)
      for (int e = c; e < E; e += G)
        for (int i = lane * 32; i < H; i += 32 * 32) prefetch_l2(p.wr + (int64_t)e * H + i);

    pdl_wait();
    bool ok = true;
    {
      // ---- top-k of every token (every CTA computes the same selection) ----
      for (int t = 0; t < T && ok; ++t) {
        if (do_route) {
          // The router CTAs store each logit with a tag in the word's high
          // half (one single-copy-atomic 64-bit store, no fence), into
          // kLogitCopies copies so that each copy's lines are polled by a
          // few CTAs only: poll this CTA's copy until every one of the
          // token's E words carries the tag, with a pause between rounds
          // (bounded).
          float lraw[kNloc];
          bool have = false;
          for (uint32_t poll = 0; poll < kSpinLimit && !have; ++poll) {
            bool mine = true;
#pragma unroll
            for (int i = 0; i < kNloc; ++i) {
              const int e = lane + 32 * i;
              lraw[i] = -FLT_MAX;
              if (e < E) {
                const unsigned long long w =
                    ld_relaxed_u64(&L.rlog[((c % kLogitCopies) * kFusedMaxTokens + t) * E + e]);
                mine &= (uint32_t)(w >> 32) == kLogitTag;
                lraw[i] = __uint_as_float((uint32_t)w);
              }
            }
            have = __all_sync(0xffffffffu, mine);
            if (!have) __nanosleep(128);
          }
          if (!have) {
            ok = false;
            break;
          }
          // selection key: the logit (any bias already added), or in
          // selection mode the sigmoid score plus the bias
          float v[kNloc];
#pragma unroll
          for (int i = 0; i < kNloc; ++i) {
            const int e = lane + 32 * i;
            float l = lraw[i];
            if (L.sel_bias && e < E) {
              l = 1.0f / (1.0f + expf(-l));
              if (p.bias) l += p.bias[(int64_t)t * p.bstride + e];
            }
            v[i] = (l == l) ? l : -FLT_MAX;  // NaN never wins
          }
          // k rounds of a warp arg-max on order-preserving integer keys:
          // one redux for the largest key, one for the lowest expert id
          // holding it (equal logits go to the lower id)
          uint32_t key[kNloc];
#pragma unroll
          for (int i = 0; i < kNloc; ++i) key[i] = lane + 32 * i < E ? float_order_key(v[i]) : 0u;
          unsigned taken = 0;
          uint32_t my_key = 0;
          int my_id = 0;
          const int nloc = (E + 31) >> 5;  // logits per lane
#pragma unroll 1  // unrolled, this once-per-call loop costs more instruction fetch than it saves
          for (int j = 0; j < K; ++j) {
            uint32_t lk = 0;
            int li = 0;
#pragma unroll
            for (int i = 0; i < kNloc; ++i)
              if (i < nloc && !((taken >> i) & 1u) && key[i] > lk) {
                lk = key[i];
                li = i;
              }
            const uint32_t m = __reduce_max_sync(0xffffffffu, lk);
            const int bid =
                (int)__reduce_min_sync(0xffffffffu, lk == m ? (uint32_t)(lane + 32 * li) : 0xffffffffu);
            if ((bid & 31) == lane) taken |= 1u << (bid >> 5);
            if (lane == j) {
              my_id = bid;
              my_key = m;
            }
          }
          // the k scores in parallel, lane j holding the j-th (selection
          // mode: from the winner's unbiased logit)
          float my_l = float_from_order_key(my_key);
          if (L.sel_bias) {
            float wl = -FLT_MAX;  // the winner's logit, from the lane that holds it
#pragma unroll
            for (int i = 0; i < kNloc; ++i) {
              const float li = __shfl_sync(0xffffffffu, lraw[i], my_id & 31);
              if (i == (my_id >> 5)) wl = li;
            }
            if (lane < K) my_l = (wl == wl) ? wl : -FLT_MAX;
          }
          const float my_s = lane < K ? 1.0f / (1.0f + expf(-my_l)) : 0.f;
          const float ssum = warp_sum(my_s);
          if (lane < K) {
            const float wgt = L.scale * my_s / ssum;
            sel_id[t][lane] = my_id;
            sel_w[t][lane] = wgt;
            if (c == 0) {
              p.ids_out[(int64_t)t * K + lane] = my_id;
              p.w_out[(int64_t)t * K + lane] = wgt;
            }
          }
        } else if (lane < K) {
          const int id = p.ids_in[(int64_t)t * K + lane];
          const bool valid = id >= 0 && id < E;
          if (!valid && c == 0) atomicOr(L.err, kErrBadId);
          sel_id[t][lane] = valid ? id : -1;
          sel_w[t][lane] = p.w_in[(int64_t)t * K + lane];
        }
      }
      if (!ok && lane == 0) {
        atomicOr(&status, 1);
        atomicOr(L.err, kErrTimeout);
      }
    }
    if (ok) {
      __syncwarp();
      // ---- route plan: routes sorted by (expert, token), by rank ----
      const int R = T * K;
      const int sb0 = S ? T : 0;
      int key[2], tk[2], ids[2];
      float wv[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int r = lane + 32 * h;
        key[h] = 0x7fffffff;
        tk[h] = 0;
        ids[h] = -1;
        wv[h] = 0.f;
        if (r < R) {
          tk[h] = r / K;
          ids[h] = sel_id[tk[h]][r % K];
          wv[h] = sel_w[tk[h]][r % K];
          if (ids[h] >= 0) key[h] = ids[h] * 16 + tk[h];
        }
        skey[r] = key[h];
      }
      __syncwarp();
      const unsigned v0 = __ballot_sync(0xffffffffu, key[0] != 0x7fffffff);
      const unsigned v1 = __ballot_sync(0xffffffffu, key[1] != 0x7fffffff);
      const int n_valid = __popc(v0) + __popc(v1);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        if (key[h] != 0x7fffffff) {
          int rank = 0;
          for (int m = 0; m < R; ++m) rank += skey[m] < key[h];
          r_tok[sb0 + rank] = tk[h];
          r_w[sb0 + rank] = wv[h];
          sorted_id[rank] = ids[h];
        }
      }
      __syncwarp();
      bool st[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int rk = lane + 32 * h;
        st[h] = rk < n_valid && (rk == 0 || sorted_id[rk - 1] != sorted_id[rk]);
      }
      const unsigned b0 = __ballot_sync(0xffffffffu, st[0]);
      const unsigned b1 = __ballot_sync(0xffffffffu, st[1]);
      const unsigned le = (2u << lane) - 1u;  // lanes <= this one
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int rk = lane + 32 * h;
        if (rk < n_valid && st[h]) {
          const int a = S - 1 + (h == 0 ? __popc(b0 & le) : __popc(b0) + __popc(b1 & le));
          ex_id[a] = sorted_id[rk];
          ex_rs[a] = sb0 + rk;
        }
      }
      const int nex = S + __popc(b0) + __popc(b1);
      if (lane == 0) {
        n_ex = nex;
        ex_rs[nex] = sb0 + n_valid;
      }
      __syncwarp();  // ex_id / ex_rs / n_ex of every lane
      if (lane == 0) {
        // The items come first, counted in a register: this CTA's share of
        // the routed up/gate rows, then its W_down rows.  Their loads go out
        // at once, before the rest of the plan.
        int ni = n_items;
        const int D = nex - S;
        const unsigned N = (unsigned)D * (unsigned)Fp;
        const int fb = (int)((unsigned)c * N / uG), fe = (int)((unsigned)(c + 1) * N / uG);
        for (int a = S; a < nex; ++a) {
          const int lo = (a - S) * Fp, hi = lo + Fp;
          int f = max(fb, lo) - lo;
          const int f_end = min(fe, hi) - lo;
          while (f < f_end && ni < kMaxItems) {
            const int grp_end = (f / kGroupRows + 1) * kGroupRows;
            const int cnt = min(min(f_end, grp_end) - f, p.fpi);
            items[ni++] = Item{0, (int16_t)a, f, cnt};
            f += cnt;
          }
        }
        for (int a = 0; a < nex && ni < kMaxItems; ++a) items[ni++] = Item{1, (int16_t)a, n0, nrows};
        n_items = ni;
        if (issued < ni && issued < nst) issue(issued++);  // the first routed rows at once
      }
      for (int idx = lane; idx < (nex - S) * T; idx += 32) {  // route of token t in expert a
        const int a = S + idx / T, t = idx % T;
        int r = -1;
        for (int sl = ex_rs[a]; sl < ex_rs[a + 1]; ++sl)
          if (r_tok[sl] == t) r = sl - ex_rs[a];
        rid[a][t] = (int8_t)r;
      }
    }
    __syncwarp();
    named_arrive(kBarPlan, kThreads);  // the tables above are visible to the consumers
    if (lane == 0) {
      int i = issued;
      for (; i < n_items; ++i) {
        const int s = stage_of(i);  // a stage's first use needs no wait
        // a spinning wait: a suspended one wakes up late, and every copy
        // issued late is a copy the consumers wait for
        if (i >= nst && !mbar_wait_ns(&empty_bar[s], (uint32_t)(round_of(i) - 1) & 1u, kWaitNs)) {
          atomicOr(&status, 2);
          break;
        }
        issue(i);
      }
      n_issued = i;
    }
  } else {
    // =========================== consumer warps ===========================
    const int ct = tid;  // 0 .. kConsumers-1
    pdl_wait();  // x, workspace, outputs and the sync words may come from the previous grid
    // the compile-time Xing4 instance takes bf16 x only (no fp32 code to fetch)
    const bool x_staged = NP > 0 || p.x_bf16 != 0;
    if (x_staged) {  // one round of 16-byte loads into the xq region (row stride Hp)
      const int h8 = H / 8, hp8 = NP > 0 ? NP * 64 : Hp / 8;
      for (int j0 = ct; j0 < T * hp8; j0 += 4 * kConsumers) {
        uint4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int j = j0 + u * kConsumers;
          const int t = j / hp8, c8 = j % hp8;
          v[u] = make_uint4(0, 0, 0, 0);
          if (j < T * hp8 && c8 < h8) v[u] = reinterpret_cast<const uint4 *>(p.x)[(int64_t)t * h8 + c8];
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int j = j0 + u * kConsumers;
          if (j < T * hp8) reinterpret_cast<uint4 *>(xq)[j] = v[u];
        }
      }
    }
    named_sync(kBarConsumers, kConsumers);

    // ---- router logit(s) of the experts this CTA owns ----
    if (do_route && c < E) {
      const float *wrow = reinterpret_cast<const float *>(ring + (size_t)(nst - 1) * kStage);
      if (p.wr_rows_smem > 0 && !mbar_wait_bounded(&wr_bar, 0, kPollLimit)) atomicOr(&status, 2);
      int r = 0;
      for (int e = c; e < E; e += G, ++r) {
        float acc[TT];
#pragma unroll
        for (int t = 0; t < TT; ++t) acc[t] = 0.f;
        const float *w = p.wr_rows_smem > 0 ? wrow + (size_t)r * H : p.wr + (int64_t)e * H;
        const uint16_t *xs = reinterpret_cast<const uint16_t *>(xq);
#pragma unroll 4
        for (int i = ct; i < H; i += kConsumers) {
          const float wv = w[i];
#pragma unroll
          for (int t = 0; t < TT; ++t)
            if (t < T) {
              const float xv = x_staged ? __uint_as_float((uint32_t)xs[(size_t)t * Hp + i] << 16)
                                        : load_x(p.x, 0, (int64_t)t * H + i);
              acc[t] = fmaf(xv, wv, acc[t]);
            }
        }
#pragma unroll
        for (int t = 0; t < TT; ++t) {
          const float v = warp_sum(acc[t]);
          if (lane == 0) red[warp][t] = v;
        }
        named_sync(kBarConsumers, kConsumers);
        if (warp == 0 && lane < T) {  // token `lane`: the warp partials added in warp order
          float v = red[0][lane];
          for (int w = 1; w < kConsumerWarps; ++w) v += red[w][lane];
          if (p.bias && !L.sel_bias) v += p.bias[(int64_t)lane * p.bstride + e];
          // value and tag in one word: the readers need no other ordering
          for (int r = 0; r < kLogitCopies; ++r)
            st_relaxed_u64(&L.rlog[(r * kFusedMaxTokens + lane) * E + e],
                           ((unsigned long long)kLogitTag << 32) | __float_as_uint(v));
        }
        named_sync(kBarConsumers, kConsumers);  // `red` is reused by the next expert
      }
    }
    named_sync(kBarConsumers, kConsumers);  // router done with the raw x

    // ---- quantise x in place: four threads per 32-element block, eight
    // elements each, the block maximum taken over the four by shuffles ----
    const int nq = T * hb * 4;
    for (int base = 0; base < nq; base += kConsumers) {
      const int j = base + ct, blk = j >> 2, t = blk / hb, b = blk % hb, e0 = b * 32 + (j & 3) * 8;
      float v[8];
      if (x_staged) {
        const uint4 w =
            j < nq ? *reinterpret_cast<const uint4 *>(xq + (size_t)t * Hp + e0) : make_uint4(0, 0, 0, 0);
        const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          v[2 * m] = __uint_as_float(ww[m] << 16);
          v[2 * m + 1] = __uint_as_float(ww[m] & 0xFFFF0000u);
        }
      } else {
#pragma unroll
        for (int k = 0; k < 8; ++k)
          v[k] = j < nq && e0 + k < H ? load_x(p.x, 0, (int64_t)t * H + e0 + k) : 0.f;
      }
      float m = 0.f;
#pragma unroll
      for (int k = 0; k < 8; ++k) m = fmaxf(m, fabsf(v[k]));
      m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
      m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
      if (j < nq) {
        const float sc = act_block_scale(m);
        const float inv = __uint_as_float((uint32_t)(254u << 23) - __float_as_uint(sc));
        uint32_t packed[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int q0 = max(-32767, min(32767, __float2int_rn(v[2 * k] * inv)));
          const int q1 = max(-32767, min(32767, __float2int_rn(v[2 * k + 1] * inv)));
          packed[k] = (uint32_t)(q0 & 0xFFFF) | ((uint32_t)q1 << 16);
        }
        *reinterpret_cast<uint4 *>(xq + (size_t)t * Hp + e0) =
            make_uint4(packed[0], packed[1], packed[2], packed[3]);
        if ((j & 3) == 0) sx[(size_t)t * hb + b] = sc;
      }
    }
    named_sync(kBarConsumers, kConsumers);

    // One up/gate item (gate rows of up to fpi outputs in the stage's first
    // half, their up rows in the second) is taken by one group of 8 consumer
    // warps -- items rotate among the kItemGroups groups, so that many items
    // are in work at once.  Warp w computes both rows of output f0 + (w % 8):
    // every activation load serves the gate and the up row, and SwiGLU is
    // applied inside the warp.  Each of the 8 warps arrives kItemGroups times
    // on the stage's "empty" barrier (its count is all the consumer warps).
    auto process_upgate = [&](int i) {
      const Item it = items[i];
      const int s = stage_of(i);
      if (!mbar_wait_suspend(&full_bar[s], (uint32_t)round_of(i) & 1u, kWaitNs)) atomicOr(&status, 2);
      const int rs = ex_rs[it.a], nr = ex_rs[it.a + 1] - rs;
      const int fl = warp % kGroupWarps;
      float accg[TT], accu[TT];
#pragma unroll
      for (int r = 0; r < TT; ++r) accg[r] = accu[r] = 0.f;
      if (fl < it.count) {
        const uint8_t *rowg = ring + (size_t)s * kStage + (size_t)fl * rb;
        const uint8_t *rowu = rowg + (size_t)p.fpi * rb;
        int toks[TT];
#pragma unroll
        for (int r = 0; r < TT; ++r) toks[r] = r < nr ? r_tok[rs + r] : 0;
        if constexpr (NP > 0) {
          constexpr int kHp = NP * 512, kHb = NP * 16;
          const int lofs = (lane >> 4) * kSBBytes + 16 + ((lane >> 1) & 7) * 16 + (lane & 1) * 8;
          const int dofs = (lane >> 4) * kSBBytes + ((lane >> 1) & 7) * 2;
          const int b0 = lane >> 1;
          // fully unrolled for one or two tokens (more independent work per
          // warp); rolled for more, where a 7-fold body would leave the
          // instruction cache
#pragma unroll (TT <= 2 ? NP : 1)
          for (int k = 0; k < NP; ++k) {
            const uint2 qg = *reinterpret_cast<const uint2 *>(rowg + lofs + 2 * kSBBytes * k);
            const uint2 qu = *reinterpret_cast<const uint2 *>(rowu + lofs + 2 * kSBBytes * k);
            const float dg = __half2float(*reinterpret_cast<const __half *>(rowg + dofs + 2 * kSBBytes * k));
            const float du = __half2float(*reinterpret_cast<const __half *>(rowu + dofs + 2 * kSBBytes * k));
            uint32_t g0, g1, g2, g3, u0, u1, u2, u3;
            iq4_decode8(qg.x, g0, g1);
            iq4_decode8(qg.y, g2, g3);
            iq4_decode8(qu.x, u0, u1);
            iq4_decode8(qu.y, u2, u3);
#pragma unroll
            for (int r = 0; r < TT; ++r) {
              if (r < nr) {
                const int16_t *xr = xq + toks[r] * kHp + lane * 16 + 512 * k;
                const uint4 xa = *reinterpret_cast<const uint4 *>(xr);
                const uint4 xb = *reinterpret_cast<const uint4 *>(xr + 8);
                const float sxv = sx[toks[r] * kHb + b0 + 16 * k];
                const int sg = dot8_dp2a(g0, g1, xa, 0) + dot8_dp2a(g2, g3, xb, 0);
                const int su = dot8_dp2a(u0, u1, xa, 0) + dot8_dp2a(u2, u3, xb, 0);
                accg[r] = fmaf((float)sg, dg * sxv, accg[r]);
                accu[r] = fmaf((float)su, du * sxv, accu[r]);
              }
            }
          }
        } else {
#pragma unroll 2
          for (int pos = lane; pos < Hp / 16; pos += 32) {
            const int b = pos >> 1, sb = b >> 3, j = b & 7, half = pos & 1;
            const uint8_t *pg = rowg + sb * kSBBytes, *pu = rowu + sb * kSBBytes;
            const float dg = __half2float(reinterpret_cast<const __half *>(pg)[j]);
            const float du = __half2float(reinterpret_cast<const __half *>(pu)[j]);
            const uint2 qg = *reinterpret_cast<const uint2 *>(pg + 16 + j * 16 + half * 8);
            const uint2 qu = *reinterpret_cast<const uint2 *>(pu + 16 + j * 16 + half * 8);
            uint32_t g0, g1, g2, g3, u0, u1, u2, u3;
            iq4_decode8(qg.x, g0, g1);
            iq4_decode8(qg.y, g2, g3);
            iq4_decode8(qu.x, u0, u1);
            iq4_decode8(qu.y, u2, u3);
#pragma unroll
            for (int r = 0; r < TT; ++r) {
              if (r < nr) {
                const uint4 *xp4 = reinterpret_cast<const uint4 *>(xq + (size_t)toks[r] * Hp + pos * 16);
                const uint4 xa = xp4[0], xb = xp4[1];
                const float sxv = sx[(size_t)toks[r] * hb + b];
                const int sg = dot8_dp2a(g0, g1, xa, 0) + dot8_dp2a(g2, g3, xb, 0);
                const int su = dot8_dp2a(u0, u1, xa, 0) + dot8_dp2a(u2, u3, xb, 0);
                accg[r] = fmaf((float)sg, dg * sxv, accg[r]);
                accu[r] = fmaf((float)su, du * sxv, accu[r]);
              }
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive_cnt(&empty_bar[s], kItemGroups);  // for this warp and its idle twins
      if (fl < it.count) {
#pragma unroll
        for (int r = 0; r < TT; ++r) {
          if (r < nr) {
            const float g = warp_sum(accg[r]), u = warp_sum(accu[r]);
            if (lane == 0) L.h32[(int64_t)(rs + r) * Fp + it.f0 + fl] = g / (1.0f + expf(-g)) * u;
          }
        }
      }
    };

    // The up/gate items through one call site: the shared expert's, known
    // from the start, then the routed ones once the producer has planned
    // them -- one copy of the item code, which the shared items have
    // already brought into the instruction cache when the routed ones run.
    int i = 0, n_ug = n_shared_items;
    bool planned = false;
    const int my_group = warp / kGroupWarps;  // up/gate items rotate among the warp groups
#pragma unroll 1
    for (;; ++i) {
      if (i == n_shared_items && !planned) {
        // the producer warp plans meanwhile; a hardware barrier (it arrives
        // on every path) leaves it all the issue slots
        named_sync(kBarPlan, kThreads);
        planned = true;
        n_ug = (status & 1) ? i : n_items;
        while (n_ug > i && items[n_ug - 1].kind != 0) --n_ug;
      }
      if (i >= n_ug) break;
      if (i % kItemGroups == my_group) process_upgate(i);
    }
    if (!(status & 1)) {

      // ---- every CTA's h written ----
      named_sync(kBarConsumers, kConsumers);
      if (ct == 0) {
        red_release_add(&p.sync[1], 1u);  // every consumer's h, ordered by the barrier above
        if (!spin_until_geq(&p.sync[1], (unsigned)(G + L.barrier_slack), kSpinLimit)) {
          atomicOr(&status, 1);
          atomicOr(L.err, kErrTimeout);
        }
      }
      named_sync(kBarConsumers, kConsumers);
      pdl_launch_dependents();

      // ---- W_down rows of this CTA, summed over all experts ----
      const int npd = NPD > 0 ? NPD : Fp / 16;  // 16-weight units per row
      float acc[kUnits][TT];
#pragma unroll
      for (int m = 0; m < kUnits; ++m)
#pragma unroll
        for (int t = 0; t < TT; ++t) acc[m][t] = 0.f;
      int grp_end = -1, grp_rs = 0;  // experts [.., grp_end) have their h in hq
      for (; i < n_items; ++i) {
        const Item it = items[i];
        const int a = it.a;
        const int rs = ex_rs[a];
        if (a >= grp_end) {
          // next group of whole experts that fits hq; all its loads are issued
          // before any is used (one round trip to L2)
          if (grp_end >= 0) named_sync(kBarConsumers, kConsumers);  // previous group no longer read
          int ge = a + 1;
          while (ge < n_ex && ex_rs[ge + 1] - rs <= p.hq_cap) ++ge;
          const int f4 = NPD > 0 ? NPD * 4 : Fp / 4;
          const int total4 = (ex_rs[ge] - rs) * f4;
          const float4 *src = reinterpret_cast<const float4 *>(L.h32 + (int64_t)rs * Fp);
          // float4 loads in flight per thread: at one token, 2 cover the
          // five 1,024-wide h rows of the Xing4 layer in one pass
          constexpr int kH4 = TT == 1 ? 2 : 4;
          for (int base = 0; base < total4; base += kConsumers * kH4) {
            float4 v[kH4];
#pragma unroll
            for (int m = 0; m < kH4; ++m) {
              const int j = base + ct + m * kConsumers;
              v[m] = j < total4 ? __ldcg(src + j) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int m = 0; m < kH4; ++m) {
              const int j = base + ct + m * kConsumers;  // 8 consecutive j: one 32-block
              float mx = fmaxf(fmaxf(fabsf(v[m].x), fabsf(v[m].y)), fmaxf(fabsf(v[m].z), fabsf(v[m].w)));
              mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
              mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
              mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
              if (j < total4) {
                const float sc = act_block_scale(mx);
                const float inv = __uint_as_float((uint32_t)(254u << 23) - __float_as_uint(sc));
                const int q0 = max(-32767, min(32767, __float2int_rn(v[m].x * inv)));
                const int q1 = max(-32767, min(32767, __float2int_rn(v[m].y * inv)));
                const int q2 = max(-32767, min(32767, __float2int_rn(v[m].z * inv)));
                const int q3 = max(-32767, min(32767, __float2int_rn(v[m].w * inv)));
                reinterpret_cast<uint2 *>(hq)[j] =
                    make_uint2((uint32_t)(q0 & 0xFFFF) | ((uint32_t)q1 << 16),
                               (uint32_t)(q2 & 0xFFFF) | ((uint32_t)q3 << 16));
                if ((ct & 7) == 0) shs[j / 8] = sc * r_w[rs + j / f4];  // route weight folded in
              }
            }
          }
          grp_end = ge;
          grp_rs = rs;
          named_sync(kBarConsumers, kConsumers);
        }
        if constexpr (TT == 1 && NPD > 0) {
          // One token, and every remaining expert's h staged with its W_down
          // rows in the ring at once (the ring holds them all): one pass over
          // all of them, so a thread's units of every expert are independent
          // work in flight together instead of one item after another.
          const int n_rem = n_items - i;
          if (grp_end >= n_ex && n_rem <= nst) {
            for (int j = 0; j < n_rem; ++j)
              if (!mbar_wait_ns(&full_bar[stage_of(i + j)], (uint32_t)round_of(i + j) & 1u, kWaitNs))
                atomicOr(&status, 2);
            // this warp's units (rows ct / NPD + 12 m) that exist: a warp-uniform count,
            // so only live units are issued
            const int r0u = ct / NPD, cnt = items[i].count;
            constexpr int kRowStep = kConsumers / NPD;
            const int nu = r0u + 2 * kRowStep < cnt ? 3 : r0u + kRowStep < cnt ? 2 : r0u < cnt ? 1 : 0;
            if (nu == 2)
              down_units_t1<NPD, 2>(items + i, n_rem, ring, ex_rs, rid, hq, shs, grp_rs, ct, i, nst, acc);
            else if (nu == 3)
              down_units_t1<NPD, 3>(items + i, n_rem, ring, ex_rs, rid, hq, shs, grp_rs, ct, i, nst, acc);
            else if (nu == 1)
              down_units_t1<NPD, 1>(items + i, n_rem, ring, ex_rs, rid, hq, shs, grp_rs, ct, i, nst, acc);
            __syncwarp();
            if (lane == 0)
              for (int j = 0; j < n_rem; ++j) mbar_arrive(&empty_bar[stage_of(i + j)]);
            i = n_items;
            break;
          }
        }
        const int hoff = rs - grp_rs;
        const int s = stage_of(i);
        if (!mbar_wait_suspend(&full_bar[s], (uint32_t)round_of(i) & 1u, kWaitNs)) atomicOr(&status, 2);
        int rids[TT];
#pragma unroll
        for (int t = 0; t < TT; ++t) rids[t] = t < T ? (int)rid[a][t] : -1;
        if constexpr (NPD > 0) {
          constexpr int kFp = NPD * 16, kDb = NPD / 16 * kSBBytes, kRowStep = kConsumers / NPD;
          static_assert(kConsumers % NPD == 0, "units of a thread share one position");
          const int pos = ct & (NPD - 1), b = pos >> 1;
          const int wofs = (b >> 3) * kSBBytes + 16 + (b & 7) * 16 + (pos & 1) * 8;
          const int dofs = (b >> 3) * kSBBytes + (b & 7) * 2;
          const uint8_t *st = ring + (size_t)s * kStage + (ct / NPD) * kDb;
#pragma unroll
          for (int m = 0; m < kUnits; ++m) {
            const int rr = ct / NPD + kRowStep * m;
            if (rr < it.count) {
              const uint2 q = *reinterpret_cast<const uint2 *>(st + kRowStep * kDb * m + wofs);
              const float d = __half2float(*reinterpret_cast<const __half *>(st + kRowStep * kDb * m + dofs));
              uint32_t c0, c1, c2, c3;
              iq4_decode8(q.x, c0, c1);
              iq4_decode8(q.y, c2, c3);
#pragma unroll
              for (int t = 0; t < TT; ++t) {
                const int r = rids[t];
                if (r >= 0) {
                  const int16_t *hr = hq + (hoff + r) * kFp + pos * 16;
                  const uint4 ha = *reinterpret_cast<const uint4 *>(hr);
                  const uint4 hb2 = *reinterpret_cast<const uint4 *>(hr + 8);
                  const int s0 = dot8_dp2a(c0, c1, ha, 0);
                  const int s1 = dot8_dp2a(c2, c3, hb2, 0);
                  acc[m][t] = fmaf((float)(s0 + s1), d * shs[(hoff + r) * (kFp / 32) + b], acc[m][t]);
                }
              }
            }
          }
        } else {
#pragma unroll
          for (int m = 0; m < kUnits; ++m) {
            const int u = ct + kConsumers * m;
            const int rr = u / npd, pos = u % npd;
            if (rr < it.count) {
              const int b = pos >> 1, sb = b >> 3, j = b & 7, half = pos & 1;
              const uint8_t *ps = ring + (size_t)s * kStage + (size_t)rr * db + sb * kSBBytes;
              const float d = __half2float(reinterpret_cast<const __half *>(ps)[j]);
              const uint2 q = *reinterpret_cast<const uint2 *>(ps + 16 + j * 16 + half * 8);
              uint32_t c0, c1, c2, c3;
              iq4_decode8(q.x, c0, c1);
              iq4_decode8(q.y, c2, c3);
#pragma unroll
              for (int t = 0; t < TT; ++t) {
                const int r = rids[t];
                if (r >= 0) {
                  const uint4 *hp4 =
                      reinterpret_cast<const uint4 *>(hq + (size_t)(hoff + r) * Fp + pos * 16);
                  const uint4 ha = hp4[0], hb2 = hp4[1];
                  const int s0 = dot8_dp2a(c0, c1, ha, 0);
                  const int s1 = dot8_dp2a(c2, c3, hb2, 0);
                  acc[m][t] = fmaf((float)(s0 + s1), d * shs[(size_t)(hoff + r) * fb32 + b], acc[m][t]);
                }
              }
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty_bar[s]);
      }
      // ---- reduce the units of each row in a fixed order and write the
      // owned output rows.  A row's npd units are consecutive in u, so each
      // group of g lanes (g = 32, or 16 when npd is an odd multiple of 16)
      // holds part of one row; the group sums go to the ring, idle once
      // every consumer is past its last stage, and are added in group order.
      named_sync(kBarConsumers, kConsumers);
      float *part = reinterpret_cast<float *>(ring);  // [units / g][TT]
      const int g = ((NPD > 0 ? NPD : npd) & 31) == 0 ? 32 : 16;
#pragma unroll
      for (int m = 0; m < kUnits; ++m) {
        const int u = ct + kConsumers * m;
#pragma unroll
        for (int t = 0; t < TT; ++t) {
          if (t < T) {
            float v = acc[m][t];
            if (g == 32) v += __shfl_xor_sync(0xffffffffu, v, 16);
            v += __shfl_xor_sync(0xffffffffu, v, 8);
            v += __shfl_xor_sync(0xffffffffu, v, 4);
            v += __shfl_xor_sync(0xffffffffu, v, 2);
            v += __shfl_xor_sync(0xffffffffu, v, 1);
            if ((lane & (g - 1)) == 0 && u / npd < nrows) part[(u / g) * TT + t] = v;
          }
        }
      }
      named_sync(kBarConsumers, kConsumers);
      const int gpr = npd / g;  // groups per row
      for (int idx = ct; idx < nrows * T; idx += kConsumers) {
        const int t = TT == 1 ? 0 : idx / nrows, rr = TT == 1 ? idx : idx % nrows;
        float v = part[(rr * gpr) * TT + t];
        for (int j = 1; j < gpr; ++j) v += part[(rr * gpr + j) * TT + t];
        const int64_t o = (int64_t)t * H + n0 + rr;
        if (p.out_bf16)
          reinterpret_cast<__nv_bfloat16 *>(p.out)[o] = __float2bfloat16_rn(v);
        else
          reinterpret_cast<float *>(p.out)[o] = v;
      }
    }
  }

  __syncthreads();
  if (tid == kProducerWarp * 32 && (status & 3)) {
    // a wait gave up, so consumers may have skipped items: the copies issued
    // into the ring (the last nst, one per stage) land before the CTA exits
    for (int j = max(0, n_issued - nst); j < n_issued; ++j)
      if (!mbar_wait_suspend(&full_bar[stage_of(j)], (uint32_t)round_of(j) & 1u, kWaitNs)) break;
  }
  if (tid == 0) {
    if (status & 2) atomicOr(L.err, kErrTimeout);
    __threadfence();
    last_cta = atomicAdd(&p.sync[2], 1u) == (unsigned)G - 1;
  }
  __syncthreads();
  if (last_cta) {  // last CTA out resets the words for the next call
    for (int j = tid; j < kLogitCopies * T * E; j += kThreads)
      L.rlog[(j / (T * E)) * kFusedMaxTokens * E + j % (T * E)] = 0ull;
    if (tid == 0) {
      p.sync[1] = 0;
      p.sync[2] = 0;
    }
    __threadfence();
  }
}

struct FusedPlan {
  int fpi, nstage, hq_cap, wr_rows_smem;
  size_t smem;
};

// Shared-memory plan for T tokens; false if the layer does not fit the
// single-launch kernel.
bool plan_fused(const Layer &L, int T, FusedPlan &fp) {
  if (T < 1 || T > kFusedMaxTokens || L.k > 8 || L.E > 256) return false;
  // the grid-wide handoffs need every CTA of the grid (one per SM) resident
  // at once; create checked that one CTA of every instance fits an SM
  if (!L.fused_resident || L.sms < 1) return false;
  const int g_sms = L.sms;
  // the kernel splits rows among the CTAs in 32-bit arithmetic
  const int64_t d_max = std::min<int64_t>((int64_t)T * L.k, L.E);
  if ((int64_t)std::max<int64_t>(L.H, d_max * L.Fp) * g_sms >= (int64_t)1 << 32) return false;
  fp.fpi = (int)std::min<int64_t>(8, kStage / (2 * L.gu_row_bytes));
  if (fp.fpi < 1) return false;
  const int rows_cta = (L.H + g_sms - 1) / g_sms;
  if (rows_cta > kMaxRowsCta || (int64_t)rows_cta * L.dn_row_bytes > kStage) return false;
  if ((int64_t)rows_cta * (L.Fp / 16) > (int64_t)kUnits * kConsumers) return false;
  const size_t per_route = (size_t)L.Fp * 2 + (size_t)(L.Fp / 32) * 4;
  const size_t fixed = (size_t)T * L.Hp * 2 + (size_t)T * (L.Hp / 32) * 4;
  const size_t limit = smem_limit_fused();
  if (fixed + (size_t)T * per_route + 3 * (size_t)kStage > limit) return false;
  // a multiple of kItemGroups stages: up/gate items rotate among the
  // consumer-warp groups, and a group's parity wait on a stage is only
  // exact when the stage's previous use was that group's too
  fp.nstage = (int)std::min<size_t>(kMaxStages, (limit - fixed - (size_t)T * per_route) / kStage);
  fp.nstage -= fp.nstage % kItemGroups;
  if (fp.nstage != 3 && fp.nstage != 6) return false;  // the kernel divides by 3 or 6 only
  const size_t left = limit - fixed - (size_t)fp.nstage * kStage;
  fp.hq_cap = (int)std::min<size_t>((size_t)T * (L.k + L.S), left / per_route);
  fp.smem = fixed + (size_t)fp.nstage * kStage + (size_t)fp.hq_cap * per_route;
  // router rows in the last stage when they fit and no shared item uses it
  const int router_rows = (L.E + g_sms - 1) / g_sms;
  const int64_t f_sh = L.Fp / g_sms + 1;
  const int shared_items = (int)(f_sh / fp.fpi + 2 + f_sh / kGroupRows);
  fp.wr_rows_smem = ((int64_t)router_rows * L.H * 4 <= kStage && shared_items <= fp.nstage - 1)
                        ? router_rows : 0;
  // item-count bound: shared + routed up/gate + one W_down item per expert
  const int64_t D = std::min<int64_t>((int64_t)T * L.k, L.E);
  const int64_t f_rt = D * L.Fp / g_sms + 1;
  const int64_t items = shared_items + (f_rt / fp.fpi + D + f_rt / kGroupRows + 2) + (D + L.S);
  return items <= kMaxItems;
}

// Raise the instance's shared-memory limit on the current device and report
// how many of its CTAs an SM holds at the largest plan (the grid needs 1).
template <int TT, int NP, int NPD>
cudaError_t prepare_tt(int *per_sm) {
  cudaError_t e = cudaFuncSetAttribute(decode_fused_kernel<TT, NP, NPD>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_limit_fused());
  if (e != cudaSuccess) return e;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(per_sm, decode_fused_kernel<TT, NP, NPD>, kThreads,
                                                       smem_limit_fused());
}

template <int TT, int NP, int NPD>
cudaError_t launch_tt(const Params &p, int grid, size_t smem, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  // programmatic serialization: the next call's prologue overlaps this
  // call's tail; cooperative (on request): started only once every CTA of
  // the grid can be resident at once, which the device-wide waits need
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeCooperative;
  attr[1].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = p.L.coop ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, decode_fused_kernel<TT, NP, NPD>, p);
}

}  // namespace

size_t smem_limit_fused() { return 232448 - 8192; }  // dynamic part; static tables take < 8 KB

cudaError_t decode_prepare(Layer &L) {
  int n[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  cudaError_t e = prepare_tt<1, 7, 64>(&n[0]);
  if (e == cudaSuccess) e = prepare_tt<1, 0, 0>(&n[1]);
  if (e == cudaSuccess) e = prepare_tt<2, 7, 64>(&n[2]);
  if (e == cudaSuccess) e = prepare_tt<2, 0, 0>(&n[3]);
  if (e == cudaSuccess) e = prepare_tt<4, 7, 64>(&n[4]);
  if (e == cudaSuccess) e = prepare_tt<4, 0, 0>(&n[5]);
  if (e == cudaSuccess) e = prepare_tt<8, 7, 64>(&n[6]);
  if (e == cudaSuccess) e = prepare_tt<8, 0, 0>(&n[7]);
  if (e != cudaSuccess) return e;
  L.fused_resident = *std::min_element(n, n + 8) >= 1 ? 1 : 0;
  return unit_decode_prepare(L);
}

bool fused_decode_supported(const Layer &L, int T) {
  FusedPlan fp;
  return plan_fused(L, T, fp);
}

cudaError_t launch_decode_fused(const Layer &L, const void *x, moe_dtype xdt, int T,
                                const float *wr, const float *bias, int64_t bstride,
                                const int32_t *ids_in, const float *w_in, int32_t *ids_out,
                                float *w_out, void *out, moe_dtype odt, cudaStream_t stream, void *x_import) {
  FusedPlan fp;
  if (!plan_fused(L, T, fp)) return cudaErrorInvalidConfiguration;
  if (T == 1 && unit_decode_supported(L))
    return launch_decode_unit(L, x, xdt, wr, bias, ids_in, w_in, ids_out, w_out, out, odt, stream, nullptr,
                              x_import);
  Params p;
  p.L = L;
  p.x = x;
  p.x_bf16 = xdt == MOE_DT_BF16;
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
  p.nstage = fp.nstage;
  p.fpi = fp.fpi;
  p.hq_cap = fp.hq_cap;
  p.wr_rows_smem = fp.wr_rows_smem;
  p.sync = L.sync;
  cudaError_t e;
  // compile-time shape for the Xing4 layer (H 3584, F 1024); any other shape
  // takes the runtime-loop instance
  const int tt = T <= 1 ? 1 : T <= 2 ? 2 : T <= 4 ? 4 : 8;
  const bool xing4 = L.Hp == 3584 && L.Fp == 1024 && L.E <= 64 && xdt == MOE_DT_BF16 &&
                     fp.nstage == xing4_stages(tt);
  if (T <= 1)
    e = xing4 ? launch_tt<1, 7, 64>(p, L.sms, fp.smem, stream) : launch_tt<1, 0, 0>(p, L.sms, fp.smem, stream);
  else if (T <= 2)
    e = xing4 ? launch_tt<2, 7, 64>(p, L.sms, fp.smem, stream) : launch_tt<2, 0, 0>(p, L.sms, fp.smem, stream);
  else if (T <= 4)
    e = xing4 ? launch_tt<4, 7, 64>(p, L.sms, fp.smem, stream) : launch_tt<4, 0, 0>(p, L.sms, fp.smem, stream);
  else
    e = xing4 ? launch_tt<8, 7, 64>(p, L.sms, fp.smem, stream) : launch_tt<8, 0, 0>(p, L.sms, fp.smem, stream);
  count_launches(1);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace moe
