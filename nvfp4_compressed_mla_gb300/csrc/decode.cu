// decode.cu -- entry points of the sparse absorbed-MLA decode and the split-K combine.
//
// Follows the Prime Inference post, section "Native NVFP4 sparse MLA decode
// kernel": rows chosen by the indexer are loaded compressed and dequantised
// on chip (no intermediate FP8 buffer in device memory), the math runs on
// FP16 operands with FP32 accumulation, and -1 slots are skipped without a
// load. The tensor-core kernel is in decode_tc.cu; one 2-CTA cluster handles
// one (query token, split of its top-k list). The post merges a token's
// partial results across the SMs of a cluster; here a batch-adaptive split
// count (the post's "adjust the cluster to the batch") spreads small batches
// over the GPU, and a combine kernel merges the splits through a workspace.
#include <math.h>

#include <atomic>

#include "decode_common.cuh"

namespace nvfp4_mla {
namespace {

using Params = DecodeParams;

// Merge the per-split partial results of one (query token, head): the
// split-K combine of partial softmax results (the post merges a token's
// partials across the SMs of a cluster; here through the workspace).
__global__ void __launch_bounds__(128) combine_kernel(const Params p) {
  const int64_t th = blockIdx.x;  // t * H + h
  const int t = static_cast<int>(th / p.num_heads), h = static_cast<int>(th % p.num_heads);
  const int S = p.num_splits;
  const float* wl = p.ws + static_cast<int64_t>(p.num_q) * S * p.num_heads * kLatent;
  float m = -INFINITY;
  bool failed = false;  // a split that gave up (its partial LSE is NaN) fails the token
  for (int s = 0; s < S; ++s) {
    const float ls = wl[(static_cast<int64_t>(t) * S + s) * p.num_heads + h];
    failed |= isnan(ls);
    m = fmaxf(m, ls);
  }
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  float tot = 0.f;
  if (failed) {
    acc[0] = acc[1] = acc[2] = acc[3] = NAN;
    tot = NAN;
  } else if (m != -INFINITY) {
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
  const float sc = failed ? 1.f : (tot > 0.f ? p.out_mult / tot : 0.f);
  const int64_t qh = static_cast<int64_t>(t) * p.num_heads + h;
  const int d = threadIdx.x * 4;
  if (p.out_fp32) {
    *reinterpret_cast<float4*>(static_cast<float*>(p.out) + qh * kLatent + d) =
        make_float4(acc[0] * sc, acc[1] * sc, acc[2] * sc, acc[3] * sc);
  } else {
    *reinterpret_cast<uint2*>(static_cast<uint16_t*>(p.out) + qh * kLatent + d) =
        make_uint2(pack_bf16x2(acc[0] * sc, acc[1] * sc), pack_bf16x2(acc[2] * sc, acc[3] * sc));
  }
  if (threadIdx.x == 0 && p.lse != nullptr)
    p.lse[qh] = failed ? NAN : (tot > 0.f ? m + lg2(tot) * kLn2 : -INFINITY);
}

// Splits per query token: enough (token, split) clusters to fill the GPU
// once (two SMs per cluster), with at least two 128-slot tiles per split and
// no split below four tiles: a split saves its share of the tiles but costs
// the combine launch and the workspace round trip, about two tiles' time.
int auto_splits(int num_q, int num_heads, int topk, int sms) {
  (void)num_heads;
  const int tiles = (topk + kTile - 1) / kTile;
  if (tiles < 4) return 1;
  const int clusters = sms / 2;
  int s = num_q >= clusters ? 1 : clusters / num_q;
  s = min(s, min(tiles / 2, 64));
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

constexpr long long kDefaultWaitCycles = 1ll << 31;  // about a second at GB300 clocks
std::atomic<long long> g_wait_cycles{kDefaultWaitCycles};

}  // namespace

long long decode_wait_cycles() { return g_wait_cycles.load(std::memory_order_relaxed); }

}  // namespace nvfp4_mla

using namespace nvfp4_mla;

extern "C" int32_t nvfp4_mla_set_wait_limit(int64_t cycles) {
  if (cycles < 0) return NVFP4_MLA_ERR_VALUE;
  g_wait_cycles.store(cycles == 0 ? kDefaultWaitCycles : static_cast<long long>(cycles),
                      std::memory_order_relaxed);
  return NVFP4_MLA_OK;
}

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
  p.wait_cycles = decode_wait_cycles();
  plan_splits(topk, num_splits ? num_splits : auto_splits(num_q, num_heads, topk, sms),
              &p.num_splits, &p.tiles_per_split, &p.num_tiles);
  const size_t need = workspace_bytes_for(num_q, num_heads, p.num_splits);
  if (need > 0) {
    if (workspace == nullptr || workspace_bytes < need) return NVFP4_MLA_ERR_WORKSPACE;
    if (!aligned16(workspace)) return NVFP4_MLA_ERR_ALIGN;
    p.ws = static_cast<float*>(workspace);
  }

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (int32_t st = launch_decode_tc(p, row_format, s)) return st;
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
    // The shape was validated just above, so SIZE_MAX here can only come from
    // the device query inside the split planning (no device, or not sm_103).
    if (need == SIZE_MAX) {
      int dev = 0, sms = 0;
      const int32_t st = current_device_checked(&dev, &sms);
      return st != NVFP4_MLA_OK ? st : NVFP4_MLA_ERR_DEVICE;
    }
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
