// Route plan: per-expert histogram, exclusive prefix sum and a stable
// permutation of the routes into expert order (PocketLLM "Xing4.0-29B-A4B:
// the design record", section 4: routes sorted by expert into a CSR table
// consumed by one grouped kernel; section 6: the counts must stay on the
// device -- a bincount whose size was read back to the host cost a device
// to host copy per layer and refused graph capture).
//
// Route r = t*k + j (token t, slot j).  The permutation orders routes by
// (expert, t, j): within an expert, routes keep their original order.  The
// shared expert is segment E and holds every token in order, weight 1.
// For the deterministic combine the kernel also writes route_pos[r], the
// position route r was given (-1 for a dropped route).
//
// One CTA of 1024 threads (32 warps).  Warp w owns a contiguous run of
// routes and walks it 32 at a time: lanes with the same expert find each
// other by ballots on the bits of the id, and a lane's rank is the number of
// equal lanes below it, so per-(warp, expert) counts and ranks are exact and in
// order.  Pass 1 counts, a scan turns counts into bases in expert-major,
// warp-minor order, pass 2 writes each route at base + rank.  Each lane
// loads 16 routes per round at once, so a pass costs one load round trip
// per 16,384 routes.  The same CTA then writes the tile lists of the
// tensor-core path (route tiles of <= 256 per expert -- <= 64 for batches of
// up to 64 tokens -- and every weight tile of each), from the offsets it
// holds in shared memory.
#include "device_utils.cuh"
#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kMaxE = 256;
constexpr int kPerLane = 16;

// Lanes of the warp holding the same expert id as this lane (ids < 256; ok =
// false joins no group): one ballot for validity and one per id bit, every
// lane voting in every ballot.
__device__ __forceinline__ unsigned same_expert_lanes(int e, bool ok) {
  unsigned peers = __ballot_sync(0xffffffffu, ok);
#pragma unroll
  for (int b = 0; b < 8; ++b) {
    const bool bit = (e >> b) & 1;
    const unsigned m = __ballot_sync(0xffffffffu, bit);
    peers &= bit ? m : ~m;
  }
  return ok ? peers : 0u;
}  // routes a lane holds per round (one load round trip)

__global__ void __launch_bounds__(1024) route_plan_kernel(
    const int32_t *__restrict__ ids, const float *__restrict__ wts, int T, int k, int E, int S,
    int *__restrict__ offsets, int *__restrict__ active, int *__restrict__ route_token,
    float *__restrict__ route_weight, unsigned *__restrict__ err, TcTile *__restrict__ ug,
    TcTile *__restrict__ dn, int *__restrict__ tile_counts, int ug_mtiles, int dn_mtiles, int max_ug,
    int max_dn, int *__restrict__ route_pos, int tile_routes) {
  __shared__ int cnt[32 * kMaxE];  // [warp][expert] counts, then bases
  __shared__ int off[kMaxE + 2];
  __shared__ int act[kMaxE + 2];
  __shared__ int tile_base[kMaxE + 2];
  __shared__ int n_act_s, n_rt_s;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int R = T * k;
  const int chunk = ((R + 31) / 32 + 31) & ~31;  // routes per warp, multiple of 32
  const int r_beg = warp * chunk;
  const int r_end = min(R, r_beg + chunk);
  const unsigned lt_mask = (1u << lane) - 1u;
  pdl_wait();  // the routes come from the previous launch
  pdl_launch_dependents();

  for (int i = tid; i < 32 * E; i += blockDim.x) cnt[i] = 0;
  __syncthreads();

  // pass 1: counts (a round = 32 * kPerLane routes of the warp, loaded at once)
  for (int base = r_beg; base < r_end; base += 32 * kPerLane) {
    int ev[kPerLane];
#pragma unroll
    for (int i = 0; i < kPerLane; ++i) {
      const int r = base + 32 * i + lane;
      ev[i] = r < r_end ? ids[r] : -2;
    }
#pragma unroll
    for (int i = 0; i < kPerLane; ++i) {
      if (base + 32 * i >= r_end) break;  // warp-uniform
      const int e = ev[i];
      const bool ok = e >= 0 && e < E;
      if (e != -2 && !ok) atomicOr(err, kErrBadId);
      const unsigned peers = same_expert_lanes(e, ok);
      if (ok && (peers & lt_mask) == 0) cnt[warp * E + e] += __popc(peers);
      __syncwarp();
    }
  }
  __syncthreads();

  // scan: bases within each expert over warps, then over experts
  if (tid < E) {
    int run = 0;
    for (int w = 0; w < 32; ++w) {
      const int c = cnt[w * E + tid];
      cnt[w * E + tid] = run;
      run += c;
    }
    off[tid] = run;  // total of expert tid, turned into its start below
  }
  __syncthreads();
  if (warp == 0) {  // expert starts, active list and route-tile bases, 32 experts at a time
    int run = 0, n_act = 0, nrt = 0;
    for (int e0 = 0; e0 < E + S; e0 += 32) {
      const int e = e0 + lane;
      int c = 0;
      if (e < E) c = off[e];
      else if (e == E && S) c = T;  // the shared expert's segment
      const bool in = e < E + S;
      // inclusive scans of the counts and of the route-tile counts
      const int ntile = (c + tile_routes - 1) / tile_routes;
      int cs = c, ts = ntile;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int a = __shfl_up_sync(0xffffffffu, cs, d), b2 = __shfl_up_sync(0xffffffffu, ts, d);
        if (lane >= d) {
          cs += a;
          ts += b2;
        }
      }
      const unsigned act_mask = __ballot_sync(0xffffffffu, in && c > 0);
      const int slot = n_act + __popc(act_mask & ((1u << lane) - 1u));
      if (in) {
        off[e] = run + cs - c;
        offsets[e] = run + cs - c;
        if (c > 0) {
          act[slot] = e;
          active[slot] = e;
          tile_base[slot] = nrt + ts - ntile;
        }
      }
      run += __shfl_sync(0xffffffffu, cs, 31);
      nrt += __shfl_sync(0xffffffffu, ts, 31);
      n_act += __popc(act_mask);
    }
    if (lane == 0) {
      off[E + S] = run;
      offsets[E + S] = run;
      active[E + S] = n_act;
      n_act_s = n_act;
      n_rt_s = nrt;
    }
  }
  __syncthreads();

  // pass 2: scatter
  for (int base = r_beg; base < r_end; base += 32 * kPerLane) {
    int ev[kPerLane];
    float wv[kPerLane];
#pragma unroll
    for (int i = 0; i < kPerLane; ++i) {
      const int r = base + 32 * i + lane;
      ev[i] = r < r_end ? ids[r] : -1;
      wv[i] = r < r_end ? wts[r] : 0.f;
    }
#pragma unroll
    for (int i = 0; i < kPerLane; ++i) {
      if (base + 32 * i >= r_end) break;  // warp-uniform
      const int r = base + 32 * i + lane;
      const int e = ev[i];
      const bool ok = e >= 0 && e < E;
      const unsigned peers = same_expert_lanes(e, ok);
      int pos = -1;  // dropped (invalid id)
      if (ok) {
        pos = off[e] + cnt[warp * E + e] + __popc(peers & lt_mask);
        route_token[pos] = r / k;
        route_weight[pos] = wv[i];
      }
      if (route_pos && r < r_end) route_pos[r] = pos;
      __syncwarp();
      if (ok && (peers & lt_mask) == 0) cnt[warp * E + e] += __popc(peers);
      __syncwarp();
    }
  }
  if (S) {
    for (int t = tid; t < T; t += blockDim.x) {
      route_token[off[E] + t] = t;
      route_weight[off[E] + t] = 1.0f;
    }
  }

  // tile lists of the tensor-core path: per active expert, route tiles of
  // <= tile_routes and per route tile every weight tile, in the active
  // order.  Entry (route tile rt, weight tile m) goes to rt * mtiles + m;
  // every thread takes entries of both lists (a binary search over the
  // active experts' first route tiles finds rt's expert), so no thread
  // writes more than a few of them.
  if (ug) {
    const int n_act = n_act_s, nrt = n_rt_s;
    if (tid == 0) tile_base[n_act] = nrt;
    __syncthreads();
    const int n_ug = nrt * ug_mtiles, n_all = n_ug + nrt * dn_mtiles;
    for (int idx = tid; idx < n_all; idx += blockDim.x) {
      const bool is_ug = idx < n_ug;
      const int k = is_ug ? idx : idx - n_ug;
      const int mt = is_ug ? ug_mtiles : dn_mtiles;
      const int rt = k / mt, m = k - rt * mt;
      int lo = 0, hi = n_act - 1;  // the last active expert whose first route tile is <= rt
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (tile_base[mid] <= rt) lo = mid;
        else hi = mid - 1;
      }
      const int e = act[lo], j = rt - tile_base[lo];
      const int beg = off[e], cntr = off[e + 1] - beg;
      const TcTile tt{e, m, beg + j * tile_routes, min(tile_routes, cntr - j * tile_routes)};
      if (is_ug) {
        if (k < max_ug) ug[k] = tt;
      } else if (k < max_dn) {
        dn[k] = tt;
      }
    }
    if (tid == 0) {
      tile_counts[0] = min(nrt * ug_mtiles, max_ug);
      tile_counts[1] = min(nrt * dn_mtiles, max_dn);
    }
  }
}

}  // namespace

cudaError_t launch_route_plan(const Layer &L, const int32_t *ids, const float *weights, int T,
                              cudaStream_t stream, bool tiles) {
  return count_and_check(launch_pdl(route_plan_kernel, dim3(1), dim3(1024), 0, stream, ids, weights, T, L.k,
                                    L.E, L.S, L.offsets, L.active, L.route_token, L.route_weight, L.err,
                                    tiles ? L.tiles_ug : nullptr, L.tiles_dn, L.tile_counts, L.Fp / 128, L.Hp / 256,
                                    tc_max_tiles(L, true), tc_max_tiles(L, false),
                                    L.deterministic ? L.route_pos : nullptr, tc_tile_routes(T)));
}

}  // namespace moe
