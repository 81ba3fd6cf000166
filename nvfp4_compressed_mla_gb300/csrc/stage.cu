// stage.cu -- the staged-dequant comparison path: selected NVFP4 rows
// re-encoded as FP8 576-byte rows in a device-memory buffer, for the FP8
// decode to read afterwards.
//
// The Prime Inference post, section "Native NVFP4 sparse MLA decode kernel",
// compares its fused kernel with a staged variant that first dequantises
// the selected rows into an FP8 temporary buffer and then runs the
// attention over that buffer; the temporary costs a device-memory write and
// read per layer. This file is that first step, so the two paths can be
// timed on the same inputs. It is HBM-bound: per selected row 352 bytes are
// read and 576 written.
//
// One warp per 32 consecutive (query token, slot) entries: each lane
// resolves one entry (index, sequence, length and block-table loads in
// parallel across the warp), then the warp converts the 32 rows four at a
// time with all four rows' loads in flight. Within a row, lane i owns latent
// block i (8 code bytes and scale byte i) and rope bytes 2i, 2i+1, so reads
// and writes are contiguous across the warp.
#include <math.h>

#include "common.cuh"

namespace nvfp4_mla {
namespace {

constexpr int kStageWarps = 8;  // 256 entries per 256-thread block
constexpr int kRowsInFlight = 4;

// One row's share of lane `lane`: 16 latent values -> E4M3(value / latent_scale)
// (16 bytes at 16 * lane), rope bytes 2 * lane, 2 * lane + 1 copied. When
// latent_scale is a power of two (kMul) the quotient is the product with its
// exact reciprocal (no rounding either way: the values are far from the fp32
// range limits), which avoids the division's instruction sequence.
template <bool kMul>
__device__ __forceinline__ float divide(float v, float latent_scale, float inv_scale) {
  return kMul ? v * inv_scale : v / latent_scale;
}

template <bool kMul>
__device__ __forceinline__ void convert_row_share(uint2 codes, uint8_t sc, uint16_t rope2,
                                                  float latent_scale, float inv_scale,
                                                  uint8_t* dst, int lane) {
  const float s = f16_bits_to_f32(
      static_cast<uint16_t>(e4m3x2_to_f16x2(static_cast<uint16_t>(sc)) & 0xFFFFu));
  uint32_t pairs[8];  // f16x2 of values (2k, 2k + 1), the even one in the low half
  {
    uint32_t fa[4], fb[4];
    e2m1x8_to_f16x8(codes.x, fa);
    e2m1x8_to_f16x8(codes.y, fb);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      pairs[k] = fa[k];
      pairs[4 + k] = fb[k];
    }
  }
  uint32_t out[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {  // output word q: E4M3 of values 4q .. 4q + 3
    uint32_t half[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint32_t v2 = pairs[2 * q + h];
      const float lo = f16_bits_to_f32(static_cast<uint16_t>(v2 & 0xFFFFu)) * s;
      const float hi = f16_bits_to_f32(static_cast<uint16_t>(v2 >> 16)) * s;
      half[h] = cvt_e4m3x2(divide<kMul>(hi, latent_scale, inv_scale),
                           divide<kMul>(lo, latent_scale, inv_scale));
    }
    out[q] = half[0] | (half[1] << 16);
  }
  *reinterpret_cast<uint4*>(dst + 16 * lane) = make_uint4(out[0], out[1], out[2], out[3]);
  *reinterpret_cast<uint16_t*>(dst + kLatent + 2 * lane) = rope2;
}

template <bool kMul>
__global__ void __launch_bounds__(kStageWarps * 32)
    stage_fp8_kernel(const int32_t* __restrict__ q_seq, const int32_t* __restrict__ topk_idx,
                     int32_t num_q, int32_t topk, const int32_t* __restrict__ block_table,
                     int32_t num_seqs, int32_t max_blocks, const int32_t* __restrict__ seq_lens,
                     int32_t page_size, const uint8_t* __restrict__ cache, int64_t num_blocks,
                     int64_t block_stride, float latent_scale, float inv_scale,
                     uint8_t* __restrict__ staged,
                     int64_t rows_per_q, int32_t* __restrict__ staged_idx,
                     int32_t* __restrict__ invalid_count) {
  const int lane = threadIdx.x & 31;
  const int64_t total = static_cast<int64_t>(num_q) * topk;
  const int64_t r0 = (static_cast<int64_t>(blockIdx.x) * kStageWarps + (threadIdx.x >> 5)) * 32;
  if (r0 >= total) return;
  // this lane's entry
  const int64_t r = r0 + lane;
  int64_t off = -1;
  int64_t dst_row = 0;
  int bad = 0;
  if (r < total) {
    const int32_t t = static_cast<int32_t>(r / topk);
    const int32_t j = static_cast<int32_t>(r - static_cast<int64_t>(t) * topk);
    const int32_t pos = __ldg(topk_idx + r);
    const int32_t b = __ldg(q_seq + t);
    const int32_t len = (b >= 0 && b < num_seqs) ? __ldg(seq_lens + b) : 0;
    off = pos == -1 ? -1
                    : resolve_row(b, pos, len, block_table, num_seqs, max_blocks, page_size,
                                  num_blocks, block_stride, kNvfp4Row);
    bad = (off < 0 && pos != -1) ? 1 : 0;
    staged_idx[r] = off >= 0 ? j : -1;
    dst_row = static_cast<int64_t>(t) * rows_per_q + j;
  }
  bad = __reduce_add_sync(0xffffffffu, bad);
  if (lane == 0 && bad > 0 && invalid_count != nullptr) atomicAdd(invalid_count, bad);
  // the warp's rows, kRowsInFlight at a time
#pragma unroll 1
  for (int k0 = 0; k0 < 32; k0 += kRowsInFlight) {
    uint2 codes[kRowsInFlight];
    uint8_t sc[kRowsInFlight];
    uint16_t rope2[kRowsInFlight];
    int64_t offs[kRowsInFlight];
#pragma unroll
    for (int u = 0; u < kRowsInFlight; ++u) {
      offs[u] = __shfl_sync(0xffffffffu, off, k0 + u);
      if (offs[u] >= 0) {
        const uint8_t* row = cache + offs[u];
        codes[u] = __ldg(reinterpret_cast<const uint2*>(row + 8 * lane));
        sc[u] = __ldg(row + kScaleOff + lane);
        rope2[u] = __ldg(reinterpret_cast<const uint16_t*>(row + kRopeOff + 2 * lane));
      }
    }
#pragma unroll
    for (int u = 0; u < kRowsInFlight; ++u) {
      const int64_t drow = __shfl_sync(0xffffffffu, dst_row, k0 + u);
      if (offs[u] >= 0)
        convert_row_share<kMul>(codes[u], sc[u], rope2[u], latent_scale, inv_scale,
                                staged + drow * kFp8Row, lane);
    }
  }
}

}  // namespace
}  // namespace nvfp4_mla

using namespace nvfp4_mla;

extern "C" int64_t nvfp4_mla_staged_rows_per_q(int32_t topk, int32_t page_size) {
  if (topk <= 0 || topk > NVFP4_MLA_MAX_TOPK || page_size <= 0 || page_size > (1 << 20)) return 0;
  return (static_cast<int64_t>(topk) + page_size - 1) / page_size * page_size;
}

extern "C" int32_t nvfp4_mla_stage_fp8(const int32_t* q_seq, const int32_t* topk_idx,
                                       int32_t num_q, int32_t topk, const int32_t* block_table,
                                       int32_t num_seqs, int32_t max_blocks_per_seq,
                                       const int32_t* seq_lens, int32_t page_size,
                                       const void* cache, int64_t num_blocks,
                                       int64_t block_stride_bytes, float latent_scale,
                                       void* staged, int32_t* staged_idx,
                                       int32_t* invalid_count, void* stream) {
  const int64_t rows_per_q = nvfp4_mla_staged_rows_per_q(topk, page_size);
  if (num_q < 0 || rows_per_q == 0) return NVFP4_MLA_ERR_SHAPE;
  if (num_q == 0) return NVFP4_MLA_OK;
  if (!q_seq || !topk_idx || !block_table || !seq_lens || !cache || !staged || !staged_idx)
    return NVFP4_MLA_ERR_NULL;
  if (num_seqs <= 0 || max_blocks_per_seq <= 0 || num_blocks <= 0 ||
      block_stride_bytes < static_cast<int64_t>(page_size) * kNvfp4Row)
    return NVFP4_MLA_ERR_SHAPE;
  if (!aligned16(cache) || !aligned16(staged) || (block_stride_bytes & 15)) return NVFP4_MLA_ERR_ALIGN;
  if (!(isfinite(latent_scale) && latent_scale > 0.f)) return NVFP4_MLA_ERR_VALUE;
  int dev = 0, sms = 0;
  if (int32_t st = current_device_checked(&dev, &sms)) return st;
  const int64_t rows = static_cast<int64_t>(num_q) * topk;
  const int64_t blocks = (rows + kStageWarps * 32 - 1) / (kStageWarps * 32);
  if (blocks > 0x7FFFFFFF) return NVFP4_MLA_ERR_SHAPE;
  int e = 0;
  const bool pow2 = frexpf(latent_scale, &e) == 0.5f;  // exact reciprocal exists
  auto kern = pow2 ? stage_fp8_kernel<true> : stage_fp8_kernel<false>;
  kern<<<static_cast<unsigned>(blocks), kStageWarps * 32, 0, static_cast<cudaStream_t>(stream)>>>(
      q_seq, topk_idx, num_q, topk, block_table, num_seqs, max_blocks_per_seq, seq_lens,
      page_size, static_cast<const uint8_t*>(cache), num_blocks, block_stride_bytes, latent_scale,
      pow2 ? 1.0f / latent_scale : 0.0f, static_cast<uint8_t*>(staged), rows_per_q, staged_idx,
      invalid_count);
  return launch_status();
}
