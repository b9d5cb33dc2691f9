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
//
// One CTA of 1024 threads (32 warps).  Warp w owns a contiguous run of
// routes and walks it 32 at a time: lanes with the same expert find each
// other with __match_any_sync, and a lane's rank is the number of equal
// lanes below it, so per-(warp, expert) counts and ranks are exact and in
// order.  Pass 1 counts, a scan turns counts into bases in expert-major,
// warp-minor order, pass 2 writes each route at base + rank.
#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kMaxE = 256;

__global__ void __launch_bounds__(1024) route_plan_kernel(
    const int32_t *__restrict__ ids, const float *__restrict__ wts, int T, int k, int E, int S,
    int *__restrict__ offsets, int *__restrict__ active, int *__restrict__ route_token,
    float *__restrict__ route_weight, unsigned *__restrict__ err) {
  __shared__ int cnt[32 * kMaxE];  // [warp][expert] counts, then bases
  __shared__ int off[kMaxE + 2];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int R = T * k;
  const int chunk = ((R + 31) / 32 + 31) & ~31;  // routes per warp, multiple of 32
  const int r_beg = warp * chunk;
  const int r_end = min(R, r_beg + chunk);
  const unsigned lt_mask = (1u << lane) - 1u;

  for (int i = tid; i < 32 * E; i += blockDim.x) cnt[i] = 0;
  __syncthreads();

  // pass 1: counts
  for (int base = r_beg; base < r_end; base += 32) {
    const int r = base + lane;
    const bool valid = r < r_end;
    const int e = valid ? ids[r] : -1;
    const bool ok = valid && e >= 0 && e < E;
    if (valid && !ok) atomicOr(err, kErrBadId);
    const unsigned peers = __match_any_sync(0xffffffffu, ok ? e : -1);
    if (ok && (peers & lt_mask) == 0) cnt[warp * E + e] += __popc(peers);
    __syncwarp();
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
  if (tid == 0) {
    int run = 0, n_act = 0;
    for (int e = 0; e < E; ++e) {
      const int c = off[e];
      off[e] = run;
      offsets[e] = run;
      if (c > 0) active[n_act++] = e;
      run += c;
    }
    off[E] = run;
    offsets[E] = run;
    if (S) {
      offsets[E + 1] = run + T;
      if (T > 0) active[n_act++] = E;
    }
    active[E + S] = n_act;
  }
  __syncthreads();

  // pass 2: scatter
  for (int base = r_beg; base < r_end; base += 32) {
    const int r = base + lane;
    const bool valid = r < r_end;
    const int e = valid ? ids[r] : -1;
    const bool ok = valid && e >= 0 && e < E;
    const unsigned peers = __match_any_sync(0xffffffffu, ok ? e : -1);
    if (ok) {
      const int pos = off[e] + cnt[warp * E + e] + __popc(peers & lt_mask);
      route_token[pos] = r / k;
      route_weight[pos] = wts[r];
    }
    __syncwarp();
    if (ok && (peers & lt_mask) == 0) cnt[warp * E + e] += __popc(peers);
    __syncwarp();
  }
  if (S) {
    for (int t = tid; t < T; t += blockDim.x) {
      route_token[off[E] + t] = t;
      route_weight[off[E] + t] = 1.0f;
    }
  }
}

}  // namespace

cudaError_t launch_route_plan(const Layer &L, const int32_t *ids, const float *weights, int T,
                              cudaStream_t stream) {
  route_plan_kernel<<<1, 1024, 0, stream>>>(ids, weights, T, L.k, L.E, L.S, L.offsets, L.active,
                                            L.route_token, L.route_weight, L.err);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace moe
