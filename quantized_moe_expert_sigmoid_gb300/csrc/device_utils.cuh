// Device helpers: mbarriers, 1D bulk (TMA) copies, programmatic dependent
// launch controls, bounded waits, and the in-register IQ4_NL decode.
#pragma once

#include <stdint.h>

namespace moe {

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Arrive once and add `bytes` to the transaction count of the current phase.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

// Plain arrive (count 1) on the current phase.
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// Arrive `count` times at once on the current phase.
__device__ __forceinline__ void mbar_arrive_cnt(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

// Named barrier over `n` threads (a multiple of 32); id 0 is __syncthreads.
__device__ __forceinline__ void named_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for phase `parity` of `bar` to complete; gives up after `limit` polls
// (each poll may itself suspend for a hardware-defined interval) and returns
// false so the caller can record a timeout instead of hanging.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity, uint32_t limit) {
  for (uint32_t i = 0; i < limit; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}

// Bounded wait that sleeps `ns` between polls, leaving the issue slots to
// the warps that are computing; gives up after `limit` polls.
__device__ __forceinline__ bool mbar_wait_sleep(uint64_t *bar, uint32_t parity, uint32_t limit,
                                                uint32_t ns) {
  for (uint32_t i = 0; i < limit; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    __nanosleep(ns);
  }
  return false;
}

// L2 prefetch of `bytes` (a multiple of 16) from 16-byte aligned global memory.
__device__ __forceinline__ void bulk_prefetch_l2(const void *src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// Order-preserving map of a float to an unsigned key (larger float, larger
// key; -0 and +0 share a key, NaN must be filtered by the caller), and back.
__device__ __forceinline__ uint32_t float_order_key(float v) {
  const uint32_t u = __float_as_uint(v);
  const uint32_t k = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return k == 0x7FFFFFFFu ? 0x80000000u : k;
}
__device__ __forceinline__ float float_from_order_key(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Wait for phase `parity` of `bar` for at most about `budget_ns` of wall
// time (the global timer is read every 64 polls); false on timeout.
__device__ __forceinline__ bool mbar_wait_ns(uint64_t *bar, uint32_t parity, uint64_t budget_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (;;) {
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (global_ns() - t0 > budget_ns) return false;
  }
}

// Wait for phase `parity` of `bar` with the thread suspended in hardware
// between checks: each try_wait may suspend for up to `hint_ns` and returns
// as soon as the phase completes, so waiting warps take no issue slots or
// shared-memory bandwidth from the warps that compute.  Gives up (false)
// after about `budget_ns` of wall time.
__device__ __forceinline__ bool mbar_try_wait_hint(uint64_t *bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool mbar_wait_suspend(uint64_t *bar, uint32_t parity, uint64_t budget_ns) {
  if (mbar_try_wait_hint(bar, parity, 20000u)) return true;
  const uint64_t t0 = global_ns();
  for (;;) {
    if (mbar_try_wait_hint(bar, parity, 20000u)) return true;
    if (global_ns() - t0 > budget_ns) return false;
  }
}

// Arrive on named barrier `id` without waiting (`n` threads take part).
__device__ __forceinline__ void named_arrive(int id, int n) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// 1D bulk copy global -> shared, completing on `bar` (16-byte aligned
// addresses, size a multiple of 16).
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes,
                                         uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// An L2 policy that marks the lines a copy brings in as the first to evict:
// for weights streamed once per call, so that what calls reuse (kernel code,
// router rows, activations, counters) stays in L2.
__device__ __forceinline__ uint64_t l2_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// bulk_g2s with an L2 cache policy for the source lines.
__device__ __forceinline__ void bulk_g2s_hint(void *dst, const void *src, uint32_t bytes, uint64_t *bar,
                                              uint64_t pol) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(pol)
      : "memory");
}

__device__ __forceinline__ void prefetch_l2(const void *p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// Programmatic dependent launch: wait until the preceding grid in the stream
// has completed and its memory is visible / allow the next grid to launch.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Add with release semantics at GPU scope: the caller's earlier writes, and
// those ordered before it by a CTA barrier, are visible to whoever observes
// the new value with an acquire load.
__device__ __forceinline__ void red_release_add(unsigned *p, unsigned v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t ld_acquire(const unsigned *p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Relaxed 64-bit global load / store at GPU scope: single-copy atomic for an
// aligned word, and never served from a stale L1 line.
__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long *p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_relaxed_u64(unsigned long long *p, unsigned long long v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// Spin until *ctr >= target (acquire), at most `limit` polls.  Each poll is
// an L2 round trip (several hundred ns), which bounds the wait in time; no
// sleep between polls, which measured faster for the batched decode call.
// Returns false on timeout.
__device__ __forceinline__ bool spin_until_geq(const unsigned *ctr, unsigned target,
                                               uint32_t limit) {
  for (uint32_t i = 0; i < limit; ++i)
    if (ld_acquire(ctr) >= target) return true;
  return false;
}

// ---- IQ4_NL decode -----------------------------------------------------------
//
// The layer stores 4-bit labels, not the file's indices: at load time index
// i becomes label (i >> 1) + 8 * (i & 1), so labels j and j + 8 (j < 8) hold
// the table's entries 2j and 2j+1, which have the same sign.  The label
// table is therefore
//   {-127, -83, -49, -22, 1, 25, 53, 89, -104, -65, -35, -10, 13, 38, 69, 113}.
// That pairing lets a byte permute decode four labels with two 8-entry byte
// tables: PRMT's selector nibble n < 8 picks byte n, and n >= 8 yields the
// sign of byte n & 7 replicated (0x00 or 0xFF).  With
//   lo = prmt(TL, labels)  and  hi = prmt(TH, labels ^ 0x8888)
// exactly one of the two is a real table byte and the other is 0x00 or 0xFF,
// and the table bytes are chosen so that lo ^ hi is the int8 code:
//   for a negative pair: TL[j] = ~code[j], TH[j] = code[j+8] (msb 1)
//   for a positive pair: TL[j] =  code[j], TH[j] = code[j+8] (msb 0).
constexpr uint32_t kTL0 = 0x1530527Eu, kTL1 = 0x59351901u;
constexpr uint32_t kTH0 = 0xF6DDBF98u, kTH1 = 0x7145260Du;

// PTX prmt in its default mode: selector nibble i of c[15:0] picks byte
// (nibble & 7) of {b:a}; when the nibble's bit 3 is set the picked byte's
// sign bit is replicated instead.  (The CUDA __byte_perm intrinsic documents
// only the 3-bit index, so the instruction is written out.)
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
  return r;
}

// 8 labels (nibble m of q is weight m) -> two words of int8 codes:
// c0 holds weights 0..3, c1 weights 4..7 (byte m = weight m).
__device__ __forceinline__ void iq4_decode8(uint32_t q, uint32_t &c0, uint32_t &c1) {
  const uint32_t qx = q ^ 0x88888888u;
  c0 = prmt(kTL0, kTL1, q) ^ prmt(kTH0, kTH1, qx);
  c1 = prmt(kTL0, kTL1, q >> 16) ^ prmt(kTH0, kTH1, qx >> 16);
}

// Sum over 16 weights of code * xq with 16-bit activations: xp[i] holds the
// activation pair (2i, 2i+1) as two int16.
__device__ __forceinline__ int dot16_dp2a(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3,
                                          const uint32_t xp[8], int acc) {
  asm("dp2a.lo.s32.s32 %0, %1, %2, %0;" : "+r"(acc) : "r"(xp[0]), "r"(c0));
  asm("dp2a.hi.s32.s32 %0, %1, %2, %0;" : "+r"(acc) : "r"(xp[1]), "r"(c0));
  asm("dp2a.lo.s32.s32 %0, %1, %2, %0;" : "+r"(acc) : "r"(xp[2]), "r"(c1));
  asm("dp2a.hi.s32.s32 %0, %1, %2, %0;" : "+r"(acc) : "r"(xp[3]), "r"(c1));
  asm("dp2a.lo.s32.s32 %0, %1, %2, %0;" : "+r"(acc) : "r"(xp[4]), "r"(c2));
  asm("dp2a.hi.s32.s32 %0, %1, %2, %0;" : "+r"(acc) : "r"(xp[5]), "r"(c2));
  asm("dp2a.lo.s32.s32 %0, %1, %2, %0;" : "+r"(acc) : "r"(xp[6]), "r"(c3));
  asm("dp2a.hi.s32.s32 %0, %1, %2, %0;" : "+r"(acc) : "r"(xp[7]), "r"(c3));
  return acc;
}

// Sum over 8 weights (codes c0: weights 0..3, c1: 4..7) with activation
// pairs x = {(0,1), (2,3), (4,5), (6,7)} as int16x2; one dependency chain of
// four dp2a, so two of these run side by side per 16 weights.
__device__ __forceinline__ int dot8_dp2a(uint32_t c0, uint32_t c1, const uint4 &x, int acc) {
  asm("dp2a.lo.s32.s32 %0, %1, %2, %0;" : "+r"(acc) : "r"(x.x), "r"(c0));
  asm("dp2a.hi.s32.s32 %0, %1, %2, %0;" : "+r"(acc) : "r"(x.y), "r"(c0));
  asm("dp2a.lo.s32.s32 %0, %1, %2, %0;" : "+r"(acc) : "r"(x.z), "r"(c1));
  asm("dp2a.hi.s32.s32 %0, %1, %2, %0;" : "+r"(acc) : "r"(x.w), "r"(c1));
  return acc;
}

// Power-of-two block scale for 16-bit activations: for a block whose largest
// magnitude is m (> 0, finite), returns s = 2^(floor(log2 m) - 13), so that
// |v / s| < 2^14 for every v of the block.  Values whose exponent is within
// 6 of the block's largest keep all 8 bits of a bf16 mantissa exactly.
__device__ __forceinline__ float act_block_scale(float m) {
  int e = (int)((__float_as_uint(m) >> 23) & 0xFF) - 127;  // floor(log2 m) for normal m
  if (e < -100) e = -100;
  return __uint_as_float((uint32_t)(127 + e - 13) << 23);
}

}  // namespace moe
