// common.cuh -- shared host/device helpers of the NVFP4 MLA library (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "nvfp4_mla.h"

namespace nvfp4_mla {

constexpr int kLatent = NVFP4_MLA_LATENT_DIM;   // 512
constexpr int kRope = NVFP4_MLA_ROPE_DIM;       // 64
constexpr int kQK = kLatent + kRope;            // 576
constexpr int kGroup = NVFP4_MLA_SCALE_GROUP;   // 16
constexpr int kNvfp4Row = NVFP4_MLA_NVFP4_ROW_BYTES;  // 352
constexpr int kFp8Row = NVFP4_MLA_FP8_ROW_BYTES;      // 576
constexpr int kPayloadBytes = kLatent / 2;      // 256
constexpr int kScaleOff = kPayloadBytes;        // 256
constexpr int kRopeOff = kScaleOff + kLatent / kGroup;  // 288

static_assert(kPayloadBytes + kLatent / kGroup + kRope == kNvfp4Row, "352-byte NVFP4 row");
static_assert(kLatent + kRope == kFp8Row, "576-byte FP8 row");

// ------------------------------------------------------------ host side
// Current device, checked to be an sm_103 part; caches the SM count.
int32_t current_device_checked(int* device, int* num_sms);
bool aligned16(const void* p);
int32_t launch_status();  // maps cudaGetLastError to a status

// --------------------------------------------------------- device side
// Two fp32 -> packed E4M3x2, round to nearest even, saturating to +-448.
// `hi` lands in bits 15..8, `lo` in bits 7..0.
__device__ __forceinline__ uint32_t cvt_e4m3x2(float hi, float lo) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Packed E4M3x2 (16 bits) -> f16x2 (exact); byte 1 -> high half.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t v) {
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(v));
  return r;
}

// Four E2M1x2 bytes (one 32-bit word, 8 codes) -> four f16x2 words (exact).
// The low nibble of each byte becomes the low half of its f16x2 word.
__device__ __forceinline__ void e2m1x8_to_f16x8(uint32_t w, uint32_t (&h)[4]) {
  asm("{\n"
      ".reg .b8 b0, b1, b2, b3;\n"
      "mov.b32 {b0, b1, b2, b3}, %4;\n"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n"
      "cvt.rn.f16x2.e2m1x2 %1, b1;\n"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n"
      "cvt.rn.f16x2.e2m1x2 %3, b3;\n"
      "}\n"
      : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
      : "r"(w));
}

__device__ __forceinline__ float f16_bits_to_f32(uint16_t h) {  // exact widening
  float r;
  asm("cvt.f32.f16 %0, %1;" : "=f"(r) : "h"(h));
  return r;
}

__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

__device__ __forceinline__ float ex2(float x) {  // 2^x, hardware approximation
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

__device__ __forceinline__ float lg2(float x) {  // log2(x), hardware approximation
  float r;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ uint4 ld_nc_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// Resolve logical position `pos` of sequence `b` to a byte offset in the
// pool; -1 when it does not resolve. `len` < 0 skips the length check.
__device__ __forceinline__ int64_t resolve_row(int32_t b, int32_t pos, int32_t len,
                                               const int32_t* __restrict__ block_table,
                                               int32_t num_seqs, int32_t max_blocks,
                                               int32_t page_size, int64_t num_blocks,
                                               int64_t block_stride, int32_t row_bytes) {
  if (b < 0 || b >= num_seqs || pos < 0) return -1;
  if (len >= 0 && pos >= len) return -1;
  const int32_t lb = pos / page_size;
  if (lb >= max_blocks) return -1;
  const int64_t pb = __ldg(block_table + static_cast<int64_t>(b) * max_blocks + lb);
  if (pb < 0 || pb >= num_blocks) return -1;
  return pb * block_stride + static_cast<int64_t>(pos - lb * page_size) * row_bytes;
}

}  // namespace nvfp4_mla
