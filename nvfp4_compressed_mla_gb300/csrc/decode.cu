// decode.cu -- sparse absorbed-MLA decode over the paged NVFP4 (or FP8) cache.
//
// Follows the Prime Inference post, section "Native NVFP4 sparse MLA decode
// kernel": the rows chosen by the indexer are loaded compressed and
// dequantised on chip (no intermediate FP8 buffer in device memory), the
// math runs on FP16 operands with FP32 accumulation, and -1 slots of the
// position list are skipped without a load. The post's cluster-of-SMs
// split of one query token's rows becomes here a split of the top-k list
// across CTAs, merged by a small combine kernel through a workspace.
//
// Tensor-core path: mma.sync m16n8k16 (f16 x f16 -> f32).
//
// One CTA = (query token, 32-head group, split of the top-k list); 8 warps.
// Per 64-slot tile:
//   1. slot -> (sequence, position) -> page via the block table; -1 and
//      unresolvable slots are masked (the latter counted);
//   2. cp.async gathers the 352-byte rows (22 x 16 B) into a 2-stage ring,
//      one tile ahead of the math;
//   3. dequant: E2M1 codes x E4M3 scale -> FP16 (exact), E4M3 rope -> FP16;
//   4. S = Q K^T over 576 dims (warps split 2 head tiles x 4 token tiles);
//   5. online softmax in base 2 (8 threads per head row), P -> FP16;
//   6. O += P V over the 512 latent dims (each warp owns 64 of them).
#include <math.h>

#include <atomic>

#include "common.cuh"

namespace nvfp4_mla {
namespace {

constexpr int kTile = 64;
constexpr int kHeads = 32;
constexpr int kThreads = 256;
constexpr int kQStride = kQK + 8;  // halves per smem row (1168 B: rows step 4 banks)
constexpr int kSStride = kTile + 4;
constexpr int kPStride = kTile + 8;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

struct Params {
  const uint16_t* q_lat;
  const uint16_t* q_rope;
  const int32_t* q_seq;
  const int32_t* topk_idx;
  int32_t num_q, num_heads, topk;
  const int32_t* block_table;
  int32_t num_seqs, max_blocks;
  const int32_t* seq_lens;
  int32_t page_size;
  const uint8_t* cache;
  int64_t num_blocks, block_stride;
  float score_scale;  // sm_scale * log2(e)
  float q_lat_mult;   // latent_scale for FP8 rows, else 1
  float q_rope_mult;  // rope_scale
  float out_mult;     // latent_scale for FP8 rows, else 1
  void* out;
  int32_t out_fp32;
  float* lse;
  float* ws;          // [num_q, splits, H, 512] partial O, then [num_q, splits, H] lse
  int32_t num_splits, tiles_per_split, num_tiles, head_groups;
  int32_t* invalid_count;
};

template <int kFmt>
struct Layout {
  static constexpr int kRowBytes = kFmt == NVFP4_MLA_ROW_NVFP4_352 ? kNvfp4Row : kFp8Row;
  static constexpr int kQ = 0;
  static constexpr int kK = kQ + kHeads * kQStride * 2;
  static constexpr int kRaw = kK + kTile * kQStride * 2;
  static constexpr int kS = kRaw + 2 * kTile * kRowBytes;
  static constexpr int kP = kS + kHeads * kSStride * 4;
  static constexpr int kStats = kP + kHeads * kPStride * 2;  // m, l, alpha
  static constexpr int kOff = kStats + 3 * kHeads * 4;
  static constexpr int kBytes = kOff + 2 * kTile * 8;
  static_assert(kRaw % 16 == 0 && kS % 16 == 0 && kP % 16 == 0 && kOff % 8 == 0, "alignment");
};

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, "
      "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

template <int kFmt>
__global__ void __launch_bounds__(kThreads, 1) decode_mma_kernel(const Params p) {
  using L = Layout<kFmt>;
  constexpr int kRB = L::kRowBytes;
  constexpr int kChunks = kRB / 16;
  extern __shared__ __align__(128) uint8_t smem[];
  uint16_t* sQ = reinterpret_cast<uint16_t*>(smem + L::kQ);
  uint16_t* sK = reinterpret_cast<uint16_t*>(smem + L::kK);
  uint8_t* sRaw = smem + L::kRaw;
  float* sS = reinterpret_cast<float*>(smem + L::kS);
  uint16_t* sP = reinterpret_cast<uint16_t*>(smem + L::kP);
  float* sM = reinterpret_cast<float*>(smem + L::kStats);
  float* sL = sM + kHeads;
  float* sAlpha = sL + kHeads;
  int64_t* sOff = reinterpret_cast<int64_t*>(smem + L::kOff);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int64_t bid = blockIdx.x;
  const int split = static_cast<int>(bid % p.num_splits);
  bid /= p.num_splits;
  const int hg = static_cast<int>(bid % p.head_groups);
  const int t = static_cast<int>(bid / p.head_groups);
  const int h0 = hg * kHeads;
  const int32_t b = __ldg(p.q_seq + t);
  const int32_t len = (b >= 0 && b < p.num_seqs) ? __ldg(p.seq_lens + b) : 0;
  const int tile0 = split * p.tiles_per_split;
  const int tile1 = min(tile0 + p.tiles_per_split, p.num_tiles);
  const int32_t* idx_row = p.topk_idx + static_cast<int64_t>(t) * p.topk;

  // ---- Q (32 heads x 576) -> FP16 smem; scales folded into q
  for (int c = tid; c < kHeads * (kQK / 8); c += kThreads) {
    const int r = c / (kQK / 8), k = c % (kQK / 8), h = h0 + r;
    uint4 o = make_uint4(0, 0, 0, 0);
    if (h < p.num_heads) {
      const int64_t qh = static_cast<int64_t>(t) * p.num_heads + h;
      const bool lat = k < kLatent / 8;
      const uint4 v = lat ? ld_nc_v4(p.q_lat + qh * kLatent + k * 8)
                          : ld_nc_v4(p.q_rope + qh * kRope + (k - kLatent / 8) * 8);
      const float m = lat ? p.q_lat_mult : p.q_rope_mult;
      o.x = pack_f16x2(bf16_lo(v.x) * m, bf16_hi(v.x) * m);
      o.y = pack_f16x2(bf16_lo(v.y) * m, bf16_hi(v.y) * m);
      o.z = pack_f16x2(bf16_lo(v.z) * m, bf16_hi(v.z) * m);
      o.w = pack_f16x2(bf16_lo(v.w) * m, bf16_hi(v.w) * m);
    }
    *reinterpret_cast<uint4*>(sQ + r * kQStride + k * 8) = o;
  }
  if (tid < kHeads) {
    sM[tid] = -INFINITY;
    sL[tid] = 0.f;
    sAlpha[tid] = 1.f;
  }

  auto resolve = [&](int tile, int stage) {
    if (tid < kTile) {
      const int slot = tile * kTile + tid;
      int64_t off = -1;
      if (slot < p.topk) {
        const int32_t pos = __ldg(idx_row + slot);
        if (pos != -1) {
          off = resolve_row(b, pos, len, p.block_table, p.num_seqs, p.max_blocks, p.page_size,
                            p.num_blocks, p.block_stride, kRB);
          if (off < 0 && hg == 0 && p.invalid_count != nullptr) atomicAdd(p.invalid_count, 1);
        }
      }
      sOff[stage * kTile + tid] = off;
    }
  };
  auto issue = [&](int stage) {
    uint8_t* dst = sRaw + stage * kTile * kRB;
    for (int c = tid; c < kTile * kChunks; c += kThreads) {
      const int r = c / kChunks, k = c % kChunks;
      const int64_t off = sOff[stage * kTile + r];
      if (off >= 0) cp_async16(smem_u32(dst + r * kRB + k * 16), p.cache + off + k * 16);
    }
    cp_async_commit();
  };

  float o_acc[2][8][4];
#pragma unroll
  for (int i = 0; i < 2; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j)
#pragma unroll
      for (int k = 0; k < 4; ++k) o_acc[i][j][k] = 0.f;

  if (tile0 < tile1) {
    resolve(tile0, 0);
    __syncthreads();
    issue(0);
  }

  for (int tile = tile0; tile < tile1; ++tile) {
    const int stage = (tile - tile0) & 1;
    if (tile + 1 < tile1) resolve(tile + 1, stage ^ 1);
    cp_async_wait_all();
    __syncthreads();  // rows of `tile` landed; sK and sP free; next offsets visible
    if (tile + 1 < tile1) issue(stage ^ 1);

    // ---- dequant the tile into sK (FP16, [token][576])
    const uint8_t* raw = sRaw + stage * kTile * kRB;
    const int64_t* off = sOff + stage * kTile;
    for (int i = tid; i < kTile * 36; i += kThreads) {
      int r, col;
      uint32_t h[8];
      if constexpr (kFmt == NVFP4_MLA_ROW_NVFP4_352) {
        if (i < kTile * 32) {
          r = i >> 5;
          const int j = i & 31;
          col = j * kGroup;
          if (off[r] >= 0) {
            const uint2 pl = *reinterpret_cast<const uint2*>(raw + r * kRB + j * 8);
            const uint32_t sc = raw[r * kRB + kScaleOff + j];
            const uint32_t s2 = e4m3x2_to_f16x2(static_cast<uint16_t>(sc | (sc << 8)));
            uint32_t lo[4], hi[4];
            e2m1x8_to_f16x8(pl.x, lo);
            e2m1x8_to_f16x8(pl.y, hi);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              h[q] = hmul2_u32(lo[q], s2);
              h[4 + q] = hmul2_u32(hi[q], s2);
            }
          } else {
#pragma unroll
            for (int q = 0; q < 8; ++q) h[q] = 0;
          }
        } else {
          r = (i - kTile * 32) >> 2;
          const int c = (i - kTile * 32) & 3;
          col = kLatent + c * 16;
          if (off[r] >= 0) {
            const uint4 v = *reinterpret_cast<const uint4*>(raw + r * kRB + kRopeOff + c * 16);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              h[2 * q] = e4m3x2_to_f16x2(static_cast<uint16_t>(w[q] & 0xFFFFu));
              h[2 * q + 1] = e4m3x2_to_f16x2(static_cast<uint16_t>(w[q] >> 16));
            }
          } else {
#pragma unroll
            for (int q = 0; q < 8; ++q) h[q] = 0;
          }
        }
      } else {
        r = i / 36;
        const int c = i % 36;
        col = c * 16;
        if (off[r] >= 0) {
          const uint4 v = *reinterpret_cast<const uint4*>(raw + r * kRB + c * 16);
          const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            h[2 * q] = e4m3x2_to_f16x2(static_cast<uint16_t>(w[q] & 0xFFFFu));
            h[2 * q + 1] = e4m3x2_to_f16x2(static_cast<uint16_t>(w[q] >> 16));
          }
        } else {
#pragma unroll
          for (int q = 0; q < 8; ++q) h[q] = 0;
        }
      }
      uint4* dst = reinterpret_cast<uint4*>(sK + r * kQStride + col);
      dst[0] = make_uint4(h[0], h[1], h[2], h[3]);
      dst[1] = make_uint4(h[4], h[5], h[6], h[7]);
    }
    __syncthreads();

    // ---- S = Q K^T: warp -> head tile (warp >> 2), tokens 16 * (warp & 3) .. +15
    {
      const int mt = warp >> 2, nq = warp & 3;
      float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      const uint32_t a_base = smem_u32(sQ + (mt * 16 + (lane & 15)) * kQStride + (lane >> 4) * 8);
      const uint32_t b_base = smem_u32(sK + (nq * 16 + (lane & 7) + ((lane >> 4) << 3)) * kQStride +
                                       ((lane >> 3) & 1) * 8);
#pragma unroll 4
      for (int ks = 0; ks < kQK / 16; ++ks) {
        uint32_t a[4], bb[4];
        ldsm_x4(a_base + ks * 32, a);
        ldsm_x4(b_base + ks * 32, bb);
        mma16816(acc[0], a, bb[0], bb[1]);
        mma16816(acc[1], a, bb[2], bb[3]);
      }
      const int g = lane >> 2, q4 = lane & 3;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        const int col = nq * 16 + nt * 8 + 2 * q4;
        const bool v0 = off[col] >= 0, v1 = off[col + 1] >= 0;
        const float2 top = make_float2(v0 ? acc[nt][0] * p.score_scale : -INFINITY,
                                       v1 ? acc[nt][1] * p.score_scale : -INFINITY);
        const float2 bot = make_float2(v0 ? acc[nt][2] * p.score_scale : -INFINITY,
                                       v1 ? acc[nt][3] * p.score_scale : -INFINITY);
        *reinterpret_cast<float2*>(sS + (mt * 16 + g) * kSStride + col) = top;
        *reinterpret_cast<float2*>(sS + (mt * 16 + g + 8) * kSStride + col) = bot;
      }
    }
    __syncthreads();

    // ---- online softmax (base 2): 8 threads per head row, 8 columns each
    {
      const int r = tid >> 3, q8 = tid & 7;
      const float4 x0 = *reinterpret_cast<const float4*>(sS + r * kSStride + q8 * 8);
      const float4 x1 = *reinterpret_cast<const float4*>(sS + r * kSStride + q8 * 8 + 4);
      const float v[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
      float mx = v[0];
#pragma unroll
      for (int k = 1; k < 8; ++k) mx = fmaxf(mx, v[k]);
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
      const float m_old = sM[r];
      const float m_new = fmaxf(m_old, mx);
      const bool none = m_new == -INFINITY;
      const float alpha = none ? 1.f : ex2(m_old - m_new);
      uint32_t pk[4];
      float sum = 0.f;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float p0 = none ? 0.f : ex2(v[2 * k] - m_new);
        const float p1 = none ? 0.f : ex2(v[2 * k + 1] - m_new);
        pk[k] = pack_f16x2(p0, p1);
        sum += f16_bits_to_f32(static_cast<uint16_t>(pk[k] & 0xFFFFu)) +
               f16_bits_to_f32(static_cast<uint16_t>(pk[k] >> 16));
      }
      *reinterpret_cast<uint4*>(sP + r * kPStride + q8 * 8) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
      sum += __shfl_xor_sync(0xffffffffu, sum, 1);
      sum += __shfl_xor_sync(0xffffffffu, sum, 2);
      sum += __shfl_xor_sync(0xffffffffu, sum, 4);
      if (q8 == 0) {
        sM[r] = m_new;
        sL[r] = sL[r] * alpha + sum;
        sAlpha[r] = alpha;
      }
    }
    __syncthreads();

    // ---- O = alpha * O + P V: warp owns latent dims [64 warp, 64 warp + 64)
    {
      const int g = lane >> 2;
      const float al[4] = {sAlpha[g], sAlpha[g + 8], sAlpha[16 + g], sAlpha[24 + g]};
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
          o_acc[mt][nt][0] *= al[2 * mt];
          o_acc[mt][nt][1] *= al[2 * mt];
          o_acc[mt][nt][2] *= al[2 * mt + 1];
          o_acc[mt][nt][3] *= al[2 * mt + 1];
        }
      const uint32_t pa = smem_u32(sP + (lane & 15) * kPStride + (lane >> 4) * 8);
      const uint32_t vb = smem_u32(sK + ((lane & 7) + ((lane >> 3) & 1) * 8) * kQStride +
                                   warp * 64 + (lane >> 4) * 8);
#pragma unroll
      for (int kk = 0; kk < kTile / 16; ++kk) {
        uint32_t a0[4], a1[4];
        ldsm_x4(pa + kk * 32, a0);
        ldsm_x4(pa + 16 * kPStride * 2 + kk * 32, a1);
#pragma unroll
        for (int np = 0; np < 4; ++np) {
          uint32_t bb[4];
          ldsm_x4_t(vb + kk * 16 * kQStride * 2 + np * 32, bb);
          mma16816(o_acc[0][2 * np], a0, bb[0], bb[1]);
          mma16816(o_acc[0][2 * np + 1], a0, bb[2], bb[3]);
          mma16816(o_acc[1][2 * np], a1, bb[0], bb[1]);
          mma16816(o_acc[1][2 * np + 1], a1, bb[2], bb[3]);
        }
      }
    }
  }
  __syncthreads();

  // ---- epilogue: normalise, write out (single split) or the partial
  const int g = lane >> 2, q4 = lane & 3;
#pragma unroll
  for (int mt = 0; mt < 2; ++mt)
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int r = mt * 16 + g + half * 8;
      const int h = h0 + r;
      if (h >= p.num_heads) continue;
      const float l = sL[r];
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const float lse_nat = l > 0.f ? (sM[r] + lg2(l)) * kLn2 : -INFINITY;
      const int64_t qh = static_cast<int64_t>(t) * p.num_heads + h;
      if (p.num_splits == 1) {
        const float sc = inv * p.out_mult;
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
          const int d = warp * 64 + nt * 8 + 2 * q4;
          const float o0 = o_acc[mt][nt][2 * half] * sc, o1 = o_acc[mt][nt][2 * half + 1] * sc;
          if (p.out_fp32)
            *reinterpret_cast<float2*>(static_cast<float*>(p.out) + qh * kLatent + d) =
                make_float2(o0, o1);
          else
            *reinterpret_cast<uint32_t*>(static_cast<uint16_t*>(p.out) + qh * kLatent + d) =
                pack_bf16x2(o0, o1);
        }
        if (warp == 0 && q4 == 0 && p.lse != nullptr) p.lse[qh] = lse_nat;
      } else {
        const int64_t part = (static_cast<int64_t>(t) * p.num_splits + split) * p.num_heads + h;
        float* wo = p.ws + part * kLatent;
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
          const int d = warp * 64 + nt * 8 + 2 * q4;
          *reinterpret_cast<float2*>(wo + d) =
              make_float2(o_acc[mt][nt][2 * half] * inv, o_acc[mt][nt][2 * half + 1] * inv);
        }
        if (warp == 0 && q4 == 0) {
          float* wl = p.ws + static_cast<int64_t>(p.num_q) * p.num_splits * p.num_heads * kLatent;
          wl[part] = lse_nat;
        }
      }
    }
}

// Merge the per-split partial results of one (query token, head): the
// split-K combine of partial softmax results (the post merges a token's
// partials across the SMs of a cluster; here through the workspace).
__global__ void __launch_bounds__(128) combine_kernel(const Params p) {
  const int64_t th = blockIdx.x;  // t * H + h
  const int t = static_cast<int>(th / p.num_heads), h = static_cast<int>(th % p.num_heads);
  const int S = p.num_splits;
  const float* wl = p.ws + static_cast<int64_t>(p.num_q) * S * p.num_heads * kLatent;
  float m = -INFINITY;
  for (int s = 0; s < S; ++s)
    m = fmaxf(m, wl[(static_cast<int64_t>(t) * S + s) * p.num_heads + h]);
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  float tot = 0.f;
  if (m != -INFINITY) {
    for (int s = 0; s < S; ++s) {
      const int64_t part = (static_cast<int64_t>(t) * S + s) * p.num_heads + h;
      const float ls = wl[part];
      const float w = ex2((ls - m) * kLog2e);  // 0 for an empty split (ls = -inf)
      tot += w;
      if (w > 0.f) {
        const float4 v = *reinterpret_cast<const float4*>(p.ws + part * kLatent + threadIdx.x * 4);
        acc[0] += w * v.x;
        acc[1] += w * v.y;
        acc[2] += w * v.z;
        acc[3] += w * v.w;
      }
    }
  }
  const float sc = tot > 0.f ? p.out_mult / tot : 0.f;
  const int64_t qh = static_cast<int64_t>(t) * p.num_heads + h;
  const int d = threadIdx.x * 4;
  if (p.out_fp32) {
    *reinterpret_cast<float4*>(static_cast<float*>(p.out) + qh * kLatent + d) =
        make_float4(acc[0] * sc, acc[1] * sc, acc[2] * sc, acc[3] * sc);
  } else {
    *reinterpret_cast<uint2*>(static_cast<uint16_t*>(p.out) + qh * kLatent + d) =
        make_uint2(pack_bf16x2(acc[0] * sc, acc[1] * sc), pack_bf16x2(acc[2] * sc, acc[3] * sc));
  }
  if (threadIdx.x == 0 && p.lse != nullptr) p.lse[qh] = tot > 0.f ? m + lg2(tot) * kLn2 : -INFINITY;
}

int auto_splits(int num_q, int num_heads, int topk, int sms) {
  const int tiles = (topk + kTile - 1) / kTile;
  const int hg = (num_heads + kHeads - 1) / kHeads;
  const int64_t per_split = static_cast<int64_t>(num_q) * hg;
  int s = per_split >= sms ? 1 : static_cast<int>((sms + per_split - 1) / per_split);
  s = min(s, min(tiles, 64));
  return max(s, 1);
}

// Final split count: at least one tile per split, no empty split.
void plan_splits(int topk, int requested, int* splits, int* tiles_per_split, int* tiles) {
  *tiles = (topk + kTile - 1) / kTile;
  int s = max(1, min(requested, *tiles));
  *tiles_per_split = (*tiles + s - 1) / s;
  *splits = (*tiles + *tiles_per_split - 1) / *tiles_per_split;
}

bool shape_ok(int32_t num_q, int32_t num_heads, int32_t topk) {
  return num_q >= 0 && num_heads >= 1 && num_heads <= NVFP4_MLA_MAX_HEADS && topk >= 1 &&
         topk <= NVFP4_MLA_MAX_TOPK;
}

size_t workspace_bytes_for(int num_q, int num_heads, int splits) {
  if (splits <= 1) return 0;
  return static_cast<size_t>(num_q) * splits * num_heads * (kLatent + 1) * sizeof(float);
}

}  // namespace
}  // namespace nvfp4_mla

using namespace nvfp4_mla;

extern "C" int32_t sparse_mla_decode_num_splits(int32_t num_q, int32_t num_heads, int32_t topk) {
  if (!shape_ok(num_q, num_heads, topk)) return 0;
  int dev = 0, sms = 0;
  if (current_device_checked(&dev, &sms) != NVFP4_MLA_OK) return 0;
  int s, tps, tiles;
  plan_splits(topk, auto_splits(num_q, num_heads, topk, sms), &s, &tps, &tiles);
  return s;
}

extern "C" size_t sparse_mla_decode_workspace_size(int32_t num_q, int32_t num_heads, int32_t topk,
                                                   int32_t num_splits) {
  if (!shape_ok(num_q, num_heads, topk) || num_splits < 0 || num_splits > 64) return SIZE_MAX;
  int req = num_splits;
  if (req == 0) {
    req = sparse_mla_decode_num_splits(num_q, num_heads, topk);
    if (req == 0) return SIZE_MAX;
  }
  int s, tps, tiles;
  plan_splits(topk, req, &s, &tps, &tiles);
  return workspace_bytes_for(num_q, num_heads, s);
}

extern "C" int32_t sparse_mla_decode(
    const void* q_latent, const void* q_rope, const int32_t* q_seq, const int32_t* topk_idx,
    int32_t num_q, int32_t num_heads, int32_t topk, const int32_t* block_table, int32_t num_seqs,
    int32_t max_blocks_per_seq, const int32_t* seq_lens, int32_t page_size, const void* cache,
    int64_t num_blocks, int64_t block_stride_bytes, int32_t row_format, float sm_scale,
    float latent_scale, float rope_scale, void* out, int32_t out_fp32, float* lse,
    void* workspace, size_t workspace_bytes, int32_t num_splits, int32_t* invalid_count,
    void* stream) {
  const int32_t rb = nvfp4_mla_row_bytes(row_format);
  if (rb == 0) return NVFP4_MLA_ERR_FORMAT;
  if (!shape_ok(num_q, num_heads, topk) || num_splits < 0 || num_splits > 64)
    return NVFP4_MLA_ERR_SHAPE;
  if (num_q == 0) return NVFP4_MLA_OK;
  if (!q_latent || !q_rope || !q_seq || !topk_idx || !block_table || !seq_lens || !cache || !out)
    return NVFP4_MLA_ERR_NULL;
  if (num_seqs <= 0 || max_blocks_per_seq <= 0 || page_size <= 0 || page_size > (1 << 20) ||
      num_blocks <= 0 || block_stride_bytes < static_cast<int64_t>(page_size) * rb)
    return NVFP4_MLA_ERR_SHAPE;
  if (!aligned16(q_latent) || !aligned16(q_rope) || !aligned16(cache) || !aligned16(out) ||
      (block_stride_bytes & 15))
    return NVFP4_MLA_ERR_ALIGN;
  if (!isfinite(sm_scale) || !(isfinite(rope_scale) && rope_scale > 0.f) ||
      !(isfinite(latent_scale) && latent_scale > 0.f))
    return NVFP4_MLA_ERR_VALUE;
  int dev = 0, sms = 0;
  if (int32_t st = current_device_checked(&dev, &sms)) return st;

  Params p{};
  p.q_lat = static_cast<const uint16_t*>(q_latent);
  p.q_rope = static_cast<const uint16_t*>(q_rope);
  p.q_seq = q_seq;
  p.topk_idx = topk_idx;
  p.num_q = num_q;
  p.num_heads = num_heads;
  p.topk = topk;
  p.block_table = block_table;
  p.num_seqs = num_seqs;
  p.max_blocks = max_blocks_per_seq;
  p.seq_lens = seq_lens;
  p.page_size = page_size;
  p.cache = static_cast<const uint8_t*>(cache);
  p.num_blocks = num_blocks;
  p.block_stride = block_stride_bytes;
  p.score_scale = sm_scale * kLog2e;
  const bool fp8 = row_format == NVFP4_MLA_ROW_FP8_576;
  p.q_lat_mult = fp8 ? latent_scale : 1.f;
  p.q_rope_mult = rope_scale;
  p.out_mult = fp8 ? latent_scale : 1.f;
  p.out = out;
  p.out_fp32 = out_fp32 ? 1 : 0;
  p.lse = lse;
  p.invalid_count = invalid_count;
  p.head_groups = (num_heads + kHeads - 1) / kHeads;
  plan_splits(topk, num_splits ? num_splits : auto_splits(num_q, num_heads, topk, sms),
              &p.num_splits, &p.tiles_per_split, &p.num_tiles);
  const size_t need = workspace_bytes_for(num_q, num_heads, p.num_splits);
  if (need > 0) {
    if (workspace == nullptr || workspace_bytes < need) return NVFP4_MLA_ERR_WORKSPACE;
    if (!aligned16(workspace)) return NVFP4_MLA_ERR_ALIGN;
    p.ws = static_cast<float*>(workspace);
  }

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int64_t ctas = static_cast<int64_t>(num_q) * p.head_groups * p.num_splits;
  if (ctas > 0x7FFFFFFF) return NVFP4_MLA_ERR_SHAPE;
  if (fp8) {
    constexpr int smem = Layout<NVFP4_MLA_ROW_FP8_576>::kBytes;
    cudaFuncSetAttribute(decode_mma_kernel<NVFP4_MLA_ROW_FP8_576>,
                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    decode_mma_kernel<NVFP4_MLA_ROW_FP8_576><<<static_cast<unsigned>(ctas), kThreads, smem, s>>>(p);
  } else {
    constexpr int smem = Layout<NVFP4_MLA_ROW_NVFP4_352>::kBytes;
    cudaFuncSetAttribute(decode_mma_kernel<NVFP4_MLA_ROW_NVFP4_352>,
                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    decode_mma_kernel<NVFP4_MLA_ROW_NVFP4_352>
        <<<static_cast<unsigned>(ctas), kThreads, smem, s>>>(p);
  }
  if (int32_t st = launch_status()) return st;
  if (p.num_splits > 1) {
    combine_kernel<<<static_cast<unsigned>(static_cast<int64_t>(num_q) * num_heads), 128, 0, s>>>(p);
    return launch_status();
  }
  return NVFP4_MLA_OK;
}

// ------------------------------------------------------------------------
// Decode for callers that cannot allocate device memory: the split-K
// scratch is a static device array of this translation unit instead of a
// caller workspace. Its device address is looked up once per device (with
// that device current) and cached; the first call on a device therefore
// belongs before any stream capture. Concurrent calls share the array and
// race; each call writes every scratch element it later reads.
namespace nvfp4_mla {
namespace {
constexpr size_t kNoAllocScratch = NVFP4_MLA_NOALLOC_SCRATCH_BYTES;
__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratch];
constexpr int kScratchDevices = 64;
std::atomic<uintptr_t> g_noalloc_ptr[kScratchDevices];

int32_t noalloc_scratch(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kScratchDevices) {
    cudaGetLastError();
    return NVFP4_MLA_ERR_DEVICE;
  }
  uintptr_t p = g_noalloc_ptr[dev].load(std::memory_order_acquire);
  if (p == 0) {
    void* addr = nullptr;
    if (cudaGetSymbolAddress(&addr, g_noalloc_scratch) != cudaSuccess || addr == nullptr) {
      cudaGetLastError();
      return NVFP4_MLA_ERR_LAUNCH;
    }
    p = reinterpret_cast<uintptr_t>(addr);
    g_noalloc_ptr[dev].store(p, std::memory_order_release);
  }
  *out = reinterpret_cast<void*>(p);
  return NVFP4_MLA_OK;
}
}  // namespace
}  // namespace nvfp4_mla

extern "C" int32_t sparse_mla_decode_noalloc(
    const void* q_latent, const void* q_rope, const int32_t* q_seq, const int32_t* topk_idx,
    int32_t num_q, int32_t num_heads, int32_t topk, const int32_t* block_table, int32_t num_seqs,
    int32_t max_blocks_per_seq, const int32_t* seq_lens, int32_t page_size, const void* cache,
    int64_t num_blocks, int64_t block_stride_bytes, int32_t row_format, float sm_scale,
    float latent_scale, float rope_scale, void* out, int32_t out_fp32, float* lse,
    int32_t num_splits, int32_t* invalid_count, void* stream) {
  void* scratch = nullptr;
  if (num_q > 0 && shape_ok(num_q, num_heads, topk) && num_splits >= 0 && num_splits <= 64) {
    const size_t need = sparse_mla_decode_workspace_size(num_q, num_heads, topk, num_splits);
    if (need == SIZE_MAX) return NVFP4_MLA_ERR_DEVICE;
    if (need > kNoAllocScratch) return NVFP4_MLA_ERR_WORKSPACE;
    if (need > 0) {
      if (int32_t st = noalloc_scratch(&scratch)) return st;
    }
  }
  return sparse_mla_decode(q_latent, q_rope, q_seq, topk_idx, num_q, num_heads, topk, block_table,
                           num_seqs, max_blocks_per_seq, seq_lens, page_size, cache, num_blocks,
                           block_stride_bytes, row_format, sm_scale, latent_scale, rope_scale, out,
                           out_fp32, lse, scratch, scratch ? kNoAllocScratch : 0, num_splits,
                           invalid_count, stream);
}
