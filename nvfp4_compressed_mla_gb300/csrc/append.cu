// append.cu -- quantize-on-append into the paged NVFP4 (or FP8) MLA cache.
//
// Row format from the Prime Inference post, section "Making room for
// low-latency decode": the 512 latent values become 4-bit E2M1 codes with
// one E4M3 scale per 16 values, the 64 rope values stay FP8, 352 bytes per
// row. The post does not describe this kernel; it only implies it (the cache
// is NVFP4, and decode keeps adding tokens to it).
//
// One warp encodes one token: lane j owns latent block j (16 values, 32
// bytes of bf16 input, 8 bytes of codes + 1 scale byte of output) and rope
// values 2j, 2j+1. Every load is a coalesced 16-byte vector; the row is
// written as 8-byte payload stores, 1-byte scales and 2-byte rope pairs
// that together cover whole 32-byte sectors. The token's values are loaded
// before its slot is resolved, so those loads overlap the index and
// block-table loads. HBM-bound: 1152 bytes read and 352 written per token.
#include <math.h>

#include "common.cuh"

namespace nvfp4_mla {
namespace {

constexpr int kAppendWarps = 8;

// x / s rounded to fp32. For a power-of-two s the product with its exact
// reciprocal is the same correctly rounded value, without the division's
// instruction sequence.
__device__ __forceinline__ float div_scale(float x, float s, float inv_pow2) {
  return inv_pow2 != 0.f ? x * inv_pow2 : __fdiv_rn(x, s);
}

// E2M1 code of x under scale S > 0: nearest grid value of x/S, ties to the
// even code, saturating at 6, sign from x. Decided by comparing |x| with
// midpoint*S, products that are exact in fp32 (midpoints have <= 3
// significant bits, E4M3 scales <= 4), so no quotient is rounded.
__device__ __forceinline__ uint32_t e2m1_code(float x, float S) {
  const float a = fabsf(x);
  const uint32_t mag = (a > 0.25f * S) + (a >= 0.75f * S) + (a > 1.25f * S) +
                       (a >= 1.75f * S) + (a > 2.5f * S) + (a >= 3.5f * S) + (a > 5.0f * S);
  return mag | ((__float_as_uint(x) >> 31) << 3);
}

template <int kFmt>
__global__ void __launch_bounds__(kAppendWarps * 32)
    append_kernel(const uint8_t* __restrict__ latent, const uint8_t* __restrict__ rope,
                  const int32_t* __restrict__ seq_ids, const int32_t* __restrict__ positions,
                  int32_t n_tok, const int32_t* __restrict__ block_table, int32_t num_seqs,
                  int32_t max_blocks, int32_t page_size, uint8_t* __restrict__ cache,
                  int64_t num_blocks, int64_t block_stride, float latent_scale, float rope_scale,
                  float inv_latent_pow2, float inv_rope_pow2, int32_t* __restrict__ invalid_count) {
  constexpr int kRowBytes = kFmt == NVFP4_MLA_ROW_NVFP4_352 ? kNvfp4Row : kFp8Row;
  const int lane = threadIdx.x & 31;
  const int64_t t = static_cast<int64_t>(blockIdx.x) * kAppendWarps + (threadIdx.x >> 5);
  if (t >= n_tok) return;
  const uint8_t* src = latent + t * (kLatent * 2) + lane * (kGroup * 2);
  const uint4 a = ld_nc_v4(src);
  const uint4 b = ld_nc_v4(src + 16);
  const uint32_t rw = __ldg(reinterpret_cast<const uint32_t*>(rope + t * (kRope * 2)) + lane);
  const int64_t off = resolve_row(__ldg(seq_ids + t), __ldg(positions + t), -1, block_table,
                                  num_seqs, max_blocks, page_size, num_blocks, block_stride,
                                  kRowBytes);
  if (off < 0) {
    if (lane == 0 && invalid_count != nullptr) atomicAdd(invalid_count, 1);
    return;
  }
  uint8_t* row = cache + off;

  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
  float x[kGroup];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    x[2 * i] = bf16_lo(w[i]);
    x[2 * i + 1] = bf16_hi(w[i]);
  }

  if constexpr (kFmt == NVFP4_MLA_ROW_NVFP4_352) {
    float amax = 0.f;
#pragma unroll
    for (int k = 0; k < kGroup; ++k) amax = fmaxf(amax, fabsf(x[k]));
    // Scale byte: E4M3 of amax/6. The correctly rounded fp32 quotient of a
    // bf16 by 6 never sits on an E4M3 rounding midpoint unless the exact
    // quotient does, so this equals rounding the exact quotient.
    const uint32_t sc = cvt_e4m3x2(0.f, __fdiv_rn(amax, 6.0f)) & 0xFFu;
    const uint32_t sh = e4m3x2_to_f16x2(static_cast<uint16_t>(sc));
    const float S = f16_bits_to_f32(static_cast<uint16_t>(sh & 0xFFFFu));
    uint32_t lo = 0, hi = 0;
    if (S > 0.f) {
#pragma unroll
      for (int k = 0; k < 8; ++k) lo |= e2m1_code(x[k], S) << (4 * k);
#pragma unroll
      for (int k = 0; k < 8; ++k) hi |= e2m1_code(x[8 + k], S) << (4 * k);
    }
    *reinterpret_cast<uint2*>(row + lane * 8) = make_uint2(lo, hi);
    row[kScaleOff + lane] = static_cast<uint8_t>(sc);
  } else {
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t p0 = cvt_e4m3x2(div_scale(x[4 * i + 1], latent_scale, inv_latent_pow2),
                                     div_scale(x[4 * i], latent_scale, inv_latent_pow2));
      const uint32_t p1 = cvt_e4m3x2(div_scale(x[4 * i + 3], latent_scale, inv_latent_pow2),
                                     div_scale(x[4 * i + 2], latent_scale, inv_latent_pow2));
      o[i] = p0 | (p1 << 16);
    }
    *reinterpret_cast<uint4*>(row + lane * 16) = make_uint4(o[0], o[1], o[2], o[3]);
  }

  const uint32_t r8 = cvt_e4m3x2(div_scale(bf16_hi(rw), rope_scale, inv_rope_pow2),
                                 div_scale(bf16_lo(rw), rope_scale, inv_rope_pow2));
  constexpr int kRopeAt = kFmt == NVFP4_MLA_ROW_NVFP4_352 ? kRopeOff : kLatent;
  *reinterpret_cast<uint16_t*>(row + kRopeAt + lane * 2) = static_cast<uint16_t>(r8);
}

}  // namespace
}  // namespace nvfp4_mla

using namespace nvfp4_mla;

extern "C" int32_t nvfp4_mla_append(const void* latent, const void* rope, const int32_t* seq_ids,
                                    const int32_t* positions, int32_t n_tok,
                                    const int32_t* block_table, int32_t num_seqs,
                                    int32_t max_blocks_per_seq, int32_t page_size, void* cache,
                                    int64_t num_blocks, int64_t block_stride_bytes,
                                    int32_t row_format, float latent_scale, float rope_scale,
                                    int32_t* invalid_count, void* stream) {
  const int32_t rb = nvfp4_mla_row_bytes(row_format);
  if (rb == 0) return NVFP4_MLA_ERR_FORMAT;
  if (n_tok < 0) return NVFP4_MLA_ERR_SHAPE;
  if (n_tok == 0) return NVFP4_MLA_OK;
  if (!latent || !rope || !seq_ids || !positions || !block_table || !cache)
    return NVFP4_MLA_ERR_NULL;
  if (num_seqs <= 0 || max_blocks_per_seq <= 0 || page_size <= 0 || page_size > (1 << 20) ||
      num_blocks <= 0 || block_stride_bytes < static_cast<int64_t>(page_size) * rb ||
      static_cast<int64_t>(num_seqs) * max_blocks_per_seq > (int64_t{1} << 40))
    return NVFP4_MLA_ERR_SHAPE;
  if (!aligned16(latent) || !aligned16(rope) || !aligned16(cache) || (block_stride_bytes & 15))
    return NVFP4_MLA_ERR_ALIGN;
  if (!(isfinite(rope_scale) && rope_scale > 0.f)) return NVFP4_MLA_ERR_VALUE;
  if (row_format == NVFP4_MLA_ROW_FP8_576 && !(isfinite(latent_scale) && latent_scale > 0.f))
    return NVFP4_MLA_ERR_VALUE;
  int dev = 0, sms = 0;
  if (int32_t st = current_device_checked(&dev, &sms)) return st;

  const dim3 grid((n_tok + kAppendWarps - 1) / kAppendWarps);
  auto inv_pow2 = [](float v) {  // 1/v when v is a power of two (exact), else 0
    int e = 0;
    return frexpf(v, &e) == 0.5f ? 1.0f / v : 0.0f;
  };
  const float inv_l = row_format == NVFP4_MLA_ROW_FP8_576 ? inv_pow2(latent_scale) : 0.0f;
  const float inv_r = inv_pow2(rope_scale);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const auto* l = static_cast<const uint8_t*>(latent);
  const auto* r = static_cast<const uint8_t*>(rope);
  auto* c = static_cast<uint8_t*>(cache);
  if (row_format == NVFP4_MLA_ROW_NVFP4_352)
    append_kernel<NVFP4_MLA_ROW_NVFP4_352><<<grid, kAppendWarps * 32, 0, s>>>(
        l, r, seq_ids, positions, n_tok, block_table, num_seqs, max_blocks_per_seq, page_size, c,
        num_blocks, block_stride_bytes, latent_scale, rope_scale, inv_l, inv_r, invalid_count);
  else
    append_kernel<NVFP4_MLA_ROW_FP8_576><<<grid, kAppendWarps * 32, 0, s>>>(
        l, r, seq_ids, positions, n_tok, block_table, num_seqs, max_blocks_per_seq, page_size, c,
        num_blocks, block_stride_bytes, latent_scale, rope_scale, inv_l, inv_r, invalid_count);
  return launch_status();
}
