// Load-time re-layout of IQ4_NL matrices into SB rows (see moe_internal.cuh).
//
// Source block (HelloSun/xing4_0-29b-IQ4_NL_EPQ model card, "對純 NumPy"):
// an fp16 scale then 16 index bytes; weight j (0..15) is the low nibble of
// byte j and weight j+16 its high nibble.  Destination: the 8 scales of a
// superblock first, then each block's 4-bit labels with weight m in nibble m.
// A label is the table index relabelled as (i >> 1) + 8 * (i & 1), which puts
// same-sign table entries at labels j and j + 8 (see device_utils.cuh).
#include "moe_internal.cuh"

namespace moe {
namespace {

// One thread per destination superblock.
__global__ void repack_kernel(const uint8_t *__restrict__ src, int rows, int K,
                              uint8_t *__restrict__ dst, int64_t dst_row_bytes,
                              int n_sb, int row_group_stride, int row_group_offset) {
  const int64_t gid = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  if (gid >= (int64_t)rows * n_sb) return;
  const int r = (int)(gid / n_sb);
  const int sb = (int)(gid % n_sb);
  const int nblk = K / kQK;
  const int64_t drow = row_group_stride > 0
                           ? (int64_t)(r / kGroupRows) * row_group_stride + row_group_offset +
                                 r % kGroupRows
                           : r;
  uint8_t *d = dst + drow * dst_row_bytes + (int64_t)sb * kSBBytes;
  const uint8_t *s_row = src + (int64_t)r * nblk * 18;
  alignas(16) uint8_t out[kSBBytes];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int b = sb * 8 + j;
    if (b < nblk) {
      const uint8_t *blk = s_row + (int64_t)b * 18;
      out[2 * j] = blk[0];
      out[2 * j + 1] = blk[1];
      uint8_t w[32];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int lo = blk[2 + i] & 15, hi = blk[2 + i] >> 4;
        w[i] = (uint8_t)((lo >> 1) + 8 * (lo & 1));
        w[i + 16] = (uint8_t)((hi >> 1) + 8 * (hi & 1));
      }
#pragma unroll
      for (int i = 0; i < 16; ++i) out[16 + 16 * j + i] = (uint8_t)(w[2 * i] | (w[2 * i + 1] << 4));
    } else {
      out[2 * j] = 0;
      out[2 * j + 1] = 0;
#pragma unroll
      for (int i = 0; i < 16; ++i) out[16 + 16 * j + i] = 0;
    }
  }
  // destination superblocks are 16-byte aligned (row pitch and base are)
  uint4 *d4 = reinterpret_cast<uint4 *>(d);
  const uint4 *o4 = reinterpret_cast<const uint4 *>(out);
#pragma unroll
  for (int i = 0; i < kSBBytes / 16; ++i) d4[i] = o4[i];
}

}  // namespace

cudaError_t launch_repack(const uint8_t *src, int rows, int K, uint8_t *dst,
                          int64_t dst_row_bytes, int row_group_stride,
                          int row_group_offset, cudaStream_t stream) {
  const int n_sb = (K + kSBW - 1) / kSBW;
  const int64_t n = (int64_t)rows * n_sb;
  if (n == 0) return cudaSuccess;
  const int threads = 128;
  const int64_t blocks = (n + threads - 1) / threads;
  repack_kernel<<<(unsigned)blocks, threads, 0, stream>>>(src, rows, K, dst, dst_row_bytes, n_sb,
                                                           row_group_stride, row_group_offset);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace moe
