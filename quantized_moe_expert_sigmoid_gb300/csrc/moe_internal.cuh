// Internal declarations of libmoe_gb300: the layer object, the repacked
// weight layout and the launchers each kernel file provides.
//
// Weight layout held by a layer ("SB rows"): a matrix W[N x K] of IQ4_NL
// blocks is stored as N rows of K/256 superblocks of 144 bytes:
//   bytes   0..15   the 8 fp16 scales of blocks 0..7 of the superblock
//   bytes  16..143  8 x 16 bytes: block j's 32 four-bit indices, weight m of
//                   the block in nibble m (byte m/2, low nibble when m even)
// Same byte count as the 18-byte blocks (8 x 18 = 144).  A whole superblock
// is one 16-byte-aligned unit, so a row segment can be fetched with 128-bit
// or bulk (TMA) copies, and a 32-bit word holds 8 consecutive weights.
// Rows of K not a multiple of 256 are padded with zero blocks (scale 0).
//
// Per expert the gate and up matrices are interleaved in groups of 64 rows:
// row 128*g + r is gate row 64*g + r, row 128*g + 64 + r is up row 64*g + r.
// A 128-row tile therefore holds gate and up for the same 64 outputs.
// The shared expert is stored as expert index E.
#pragma once

#include <cuda.h>  // CUtensorMap
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moe_gb300.h"

namespace moe {

constexpr int kQK = 32;         // weights per IQ4_NL block
constexpr int kSBW = 256;       // weights per superblock
constexpr int kSBBytes = 144;   // bytes per superblock
constexpr int kGroupRows = 64;  // gate/up interleave group

// Largest batch the single-launch decode kernel handles.
constexpr int kFusedMaxTokens = 8;
// Largest batch of the single-launch batch kernel (2..16 tokens).
constexpr int kBatchMaxTokens = 16;
// Largest batch of the batched decode path (register dequantisation + mma.sync).
constexpr int kGemvMaxTokens = 64;
constexpr int kLogitCopies = 8;  // copies of the decode kernel's tagged router logits

// Sticky device error bits (Layer::err).
constexpr unsigned kErrBadId = 1u;
constexpr unsigned kErrTimeout = 2u;
constexpr int kStageEvents = 5;  // call start, up/gate begin, up/gate end, down end, call end
constexpr unsigned kErrOverflow = 4u;  // a value left fp16 range on the tensor-core path

// One tile of the batched tensor-core path: expert id, weight tile (128
// up/gate outputs or 256 down rows), first route row (in route order) and
// number of routes (<= 256).
struct TcTile {
  int expert, mtile, row0, count;
};

struct Layer {
  // device the layer was created on, and its SM count (read at create; every
  // kernel attribute and grid size of the layer's launches comes from them)
  int device = 0, sms = 0;
  // the single-launch decode kernel's grid (one CTA per SM) can be resident
  // all at once: checked at create from the occupancy of every instance
  int fused_resident = 0;
  // the one-token unit kernel's grid can be resident all at once (create)
  int unit_resident = 0;
  // shape
  int H, E, k, F, S;  // S = number of shared experts (0 or 1)
  float scale;
  int sel_bias;              // 1: the bias shifts expert selection only (MOE_FLAG_SELECTION_BIAS)
  int deterministic;         // 1: slot-ordered combine, no float atomics (MOE_FLAG_DETERMINISTIC)
  int coop;                  // 1: the single-launch decode kernels launch cooperatively (MOE_FLAG_COOPERATIVE)
  int max_tokens;
  int Hp, Fp;                // H and F padded to multiples of 256
  int64_t gu_row_bytes;      // Hp/256 * 144
  int64_t dn_row_bytes;      // Fp/256 * 144
  int64_t gu_expert_bytes;   // 2*Fp rows
  int64_t dn_expert_bytes;   // Hp rows
  int64_t weight_bytes;      // IQ4_NL bytes of the unpadded matrices

  // weights
  uint8_t *gu = nullptr;     // [(E+S)][2*Fp][gu_row_bytes]
  uint8_t *dn = nullptr;     // [(E+S)][Hp][dn_row_bytes]

  // workspace (sized for max_tokens at create)
  int max_routes = 0;        // max_tokens*k + S*max_tokens
  float *logits = nullptr;   // [max_tokens][E]
  int *offsets = nullptr;    // [E+S+1] segment starts in route order
  int *active = nullptr;     // [E+S+1] ids of experts with routes; [E+S] = count
  int *route_token = nullptr;   // [max_routes]
  float *route_weight = nullptr; // [max_routes]
  float *h32 = nullptr;      // [min(max_tokens, 8) * (k+S)][Fp] SwiGLU output of the decode kernel
  // one-token unit kernel (decode_unit.cu)
  float *hr = nullptr;       // [k][Fp] the selected experts' SwiGLU outputs
  float *hsh = nullptr;      // [Fp] the shared expert's SwiGLU output
  unsigned long long *useq = nullptr;  // arrival counters (exit, shared h, h of each slot), never reset
  unsigned long long *ulog = nullptr;  // [E][sms] tagged router logits, one private copy per CTA
  // single-launch batch kernel, 2..16 tokens (decode_batch.cu)
  int batch_smem_limit = 0;            // its dynamic shared-memory limit; 0: the kernel is not used
  unsigned long long *bseq = nullptr;  // exit counter, then two sets (by call parity) of per-entry counters
  unsigned long long *blog = nullptr;  // [16][E][sms] tagged router logits, one private copy per CTA
  float *bpart = nullptr;              // [routes][Fp][2] first-half gate and up sums
  float *bhq = nullptr;                // [routes][32][16] quantised h words, then [routes][32] scales
  float *out_acc = nullptr;  // [max_tokens][H] fp32 accumulator
  // deterministic combine only (else nullptr)
  float *ybuf = nullptr;     // [max_routes][Hp] weighted down outputs, route order
  int *route_pos = nullptr;  // [max_tokens*k] position of route t*k+j in route order, -1: dropped
  // dense blocks (n_experts = 1, top_k = 1): every token to expert 0 at weight 1
  int32_t *dense_ids = nullptr;  // [max_tokens] zeros
  float *dense_w = nullptr;      // [max_tokens] ones
  unsigned *err = nullptr;   // sticky device error word
  unsigned *sync = nullptr;  // [4] arrival counters of the single-launch decode kernel
  unsigned long long *rlog = nullptr;  // [kLogitCopies][kFusedMaxTokens][E] tagged router logits
  void *x_stage = nullptr, *out_stage = nullptr;  // [max_tokens][H] x 4 B each (MOE_FLAG_HOST_IO)
  int barrier_slack = 0;     // extra arrivals the decode kernel's h wait expects (test hook)

  // batched tensor-core path (T > kFusedMaxTokens)
  __half *x16 = nullptr;     // [max_routes][Hp] x rows in route order, fp16
  __half *h16 = nullptr;     // [max_routes][Fp] SwiGLU outputs, fp16
  TcTile *tiles_ug = nullptr, *tiles_dn = nullptr;
  int *tile_counts = nullptr;  // [2]
  // opt-in stage timing: kStageEvents events per call slot (see the header)
  cudaEvent_t *tev = nullptr;
  int tev_slots = 0, tev_next = 0, tev_used = 0;
  CUtensorMap map_x16, map_h16;        // activation tiles of the tensor-core path (256 rows)
  CUtensorMap map_x16_64, map_h16_64;  // ... boxes of 64 rows, for batches of <= 64 tokens
  CUtensorMap map_gu_lab, map_dn_lab;  // weight labels of one k-step
  // batched decode path (9..64 tokens)
  CUtensorMap map_gu_sb, map_dn_sb;    // one superblock column of 128 weight rows
  CUtensorMap map_gu_half;             // half an up/gate row of 8 rows (batch kernel)
  CUtensorMap map_x16_16, map_h16_16;  // activation rows in route order, 16-row boxes
  int gemv_ready = 0;                  // the layer's shape fits the batched decode path
};

// Launch with programmatic dependent launch allowed: the kernel may be
// scheduled while the previous kernel in the stream is still running, so its
// launch latency overlaps that kernel's tail.  Every kernel launched this way
// executes griddepcontrol.wait (pdl_wait) before it touches memory that an
// earlier launch writes or reads, and lets its own dependents launch early.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args &&>(args)...);
}

// Records the detail string behind moe_last_error() for the calling thread
// and returns `s` (printf-style).
moe_status report_error(moe_status s, const char *fmt, ...);

// Launch counter behind moe_launch_count(); every launcher adds its kernels.
void count_launches(int n);

// One launch counted; the launch's own error, else any pending one.
inline cudaError_t count_and_check(cudaError_t e) {
  count_launches(1);
  return e != cudaSuccess ? e : cudaGetLastError();
}

// Alignment helper.
inline bool aligned(const void *p, uintptr_t a) {
  return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0;
}

// ---- launchers (each .cu file defines its own) ---------------------------

// repack.cu: one IQ4_NL matrix [rows x K] (18-byte blocks, row-major) into
// SB rows.  dst_row(r) = (r / 64) * row_group_stride + row_group_offset + r % 64
// when row_group_stride > 0, else r.
cudaError_t launch_repack(const uint8_t *src, int rows, int K, uint8_t *dst,
                          int64_t dst_row_bytes, int row_group_stride,
                          int row_group_offset, cudaStream_t stream);

// router.cu
// Large batches split H into parts whose partial logits are summed by the
// top-k kernel in part order; `logits` holds parts * T * E floats.
constexpr int kRouterMaxParts = 8;
// Batches of up to kRouterSmallT tokens have too few 32 x 64 tiles to fill
// the GPU, so they split H into up to kRouterMaxPartsSmall parts instead.
constexpr int kRouterSmallT = 128;
constexpr int kRouterMaxPartsSmall = 32;
// Logits floats a layer of max_tokens needs for the K-split parts.
inline int64_t router_logits_floats(int max_tokens, int E) {
  const int64_t a = (int64_t)kRouterMaxParts * max_tokens;
  const int64_t b = (int64_t)kRouterMaxPartsSmall * (max_tokens < kRouterSmallT ? max_tokens : kRouterSmallT);
  return (a > b ? a : b) * E;
}
// K parts for T tokens: 1 for T <= 16 (the one-pass kernel), else enough to
// fill `sms` SMs (at most max_parts, and the small-batch or large-batch cap).
int router_parts(int T, int E, int H, int sms, int max_parts);
cudaError_t launch_router_logits(const Layer &L, const void *x, moe_dtype xdt, int T,
                                 const float *wr, float *logits, int parts, cudaStream_t stream);
// sums the parts, adds the optional bias, selects; ids/weights [T][k]
cudaError_t launch_router_topk(const Layer &L, const float *logits, int parts, const float *bias,
                               int64_t bias_stride, int T, int32_t *ids, float *weights,
                               cudaStream_t stream);

// plan.cu: histogram, prefix sum and stable permutation of the routes.
// tiles: also write the tile lists of the tensor-core path.
cudaError_t launch_route_plan(const Layer &L, const int32_t *ids, const float *weights,
                              int T, cudaStream_t stream, bool tiles);

// combine.cu: the output of the batched path.  finalize: out = round(out_acc);
// ordered: out[t] = sum over slots j in order of ybuf[route_pos[t*k+j]], then
// + ybuf[offsets[E] + t] (shared), rounded once.
cudaError_t launch_fill(float *dst, float value, int n, cudaStream_t stream);  // dst[0..n) = value
cudaError_t launch_finalize(const Layer &L, int T, void *out, moe_dtype odt,
                            cudaStream_t stream);
cudaError_t launch_combine_ordered(const Layer &L, int T, void *out, moe_dtype odt,
                                   cudaStream_t stream);

// decode_fused.cu: the whole layer in one launch for T <= kFusedMaxTokens.
// ids_in == nullptr: route inside (router_w, bias used; ids_out/w_out
// written); else the given routes are used.
size_t smem_limit_fused();
// kernel attributes and the co-residency check of every decode instance, on
// the current device (create)
cudaError_t decode_prepare(Layer &L);
bool fused_decode_supported(const Layer &L, int T);

// decode_unit.cu: the whole layer for one token, split into (expert,
// 32-output block) units; taken by launch_decode_fused at T = 1 when the
// layer's shape has an instance (H padded to 3,584 or 2,560).
cudaError_t unit_decode_prepare(Layer &L);
// Single-launch batch kernel (2..16 tokens): kernel attributes and whether
// its grid fits (create, before the buffers), its tensor map (after the
// weights are allocated), buffer sizes, and the launch.
cudaError_t batch_decode_prepare(Layer &L);
cudaError_t batch_decode_maps(Layer &L);
int batch_decode_seq_words();
int64_t batch_decode_hq_floats();
int64_t batch_decode_part_floats(const Layer &L);
int64_t batch_decode_log_words(const Layer &L);
bool batch_decode_supported(const Layer &L, int T);
cudaError_t launch_decode_batch(const Layer &L, const void *x, moe_dtype xdt, int T, const float *wr,
                                const float *bias, int64_t bstride, const int32_t *ids_in, const float *w_in,
                                int32_t *ids_out, float *w_out, void *out, moe_dtype odt, cudaStream_t stream,
                                void *x_import = nullptr);
int unit_decode_seq_words();
bool unit_decode_supported(const Layer &L);
// The layer input of one trunk step, formed inside the one-token kernel:
// r_out = r_in + delta, u = bf16(rmsnorm(r_out)), x = u (CTA 0 writes r_out
// and u; r_in and r_out must not overlap).
struct ResidStep {
  const float *r_in;
  const void *delta;   // nullable
  int delta_bf16;
  float *r_out;
  __nv_bfloat16 *u_out;
  float eps;
};
cudaError_t launch_decode_unit(const Layer &L, const void *x, moe_dtype xdt, const float *wr, const float *bias,
                               const int32_t *ids_in, const float *w_in, int32_t *ids_out, float *w_out,
                               void *out, moe_dtype odt, cudaStream_t stream, const ResidStep *rs = nullptr,
                               void *x_import = nullptr);
// x_import (one token, bf16 x in host memory): a device buffer of H bf16
// values that the one-token kernel copies x into, each CTA its share, before
// every CTA reads x from it
cudaError_t launch_decode_fused(const Layer &L, const void *x, moe_dtype xdt, int T,
                                const float *wr, const float *bias, int64_t bstride,
                                const int32_t *ids_in, const float *w_in, int32_t *ids_out,
                                float *w_out, void *out, moe_dtype odt, cudaStream_t stream,
                                void *x_import = nullptr);

// prefill_tc.cu: 2D tensor-map encoding (driver entry point resolved once).
cudaError_t encode_2d(CUtensorMap *map, CUtensorMapDataType dt, void *base, uint64_t inner,
                      uint64_t rows, uint64_t row_pitch, uint32_t box_inner, uint32_t box_rows,
                      CUtensorMapSwizzle swz);

// router_tc.cu: router logits of large bf16 batches on tcgen05 (K-partial
// sums in the same layout as launch_router_logits).  false: not applicable.
bool router_tc_supported(const Layer &L, moe_dtype xdt, int T);
cudaError_t router_tc_prepare();  // kernel attribute, on the current device (create)
int router_tc_parts(const Layer &L, int T);
cudaError_t launch_router_tc(const Layer &L, const void *x, int T, const float *wr, float *logits,
                             int parts, cudaStream_t stream);

// prefill_tc.cu: grouped GEMMs on tcgen05 for T > kFusedMaxTokens.
int tc_max_tiles(const Layer &L, bool up_gate);
int tc_tile_routes(int T);  // routes per tile: 64 for batches of <= 64 tokens, else 256
cudaError_t tc_prepare(Layer &L);  // tensor maps + kernel attributes (after workspace allocation)
// ev: nullable; the events to record before up/gate, after up/gate and after down
cudaError_t launch_prefill_tc(const Layer &L, const void *x, moe_dtype xdt, int T, cudaStream_t stream,
                              cudaEvent_t *ev = nullptr);

// gemv_mma.cu: batched decode path for kFusedMaxTokens < T <= kGemvMaxTokens
// (up/gate + SwiGLU into h16, then down into out_acc or ybuf), after the
// route plan and gather_x16.  ev: nullable, as for launch_prefill_tc.
bool gemv_mma_supported(const Layer &L, int T);
cudaError_t gemv_prepare(Layer &L);  // tensor maps + kernel attributes (create)
cudaError_t launch_gemv_mma(const Layer &L, cudaStream_t stream, cudaEvent_t *ev = nullptr);
// prefill_tc.cu: x rows in route order as fp16 (x16)
// Also clears the fp32 output accumulator (T x H) unless the layer combines
// deterministically (the batched paths add into it with atomics).
cudaError_t launch_gather_x16(const Layer &L, const void *x, moe_dtype xdt, int T, cudaStream_t stream);

// norm.cu
// r_out = r_in + delta (delta may be NULL; r_out may be r_in), u = bf16(rmsnorm(r_out))
cudaError_t launch_residual_rmsnorm(const float *resid_in, const void *delta, moe_dtype ddt, float *resid_out,
                                    void *u, int T, int H, float eps, cudaStream_t stream);

}  // namespace moe
