// decode_common.cuh -- parameters shared by the decode kernel and its entry point.
#pragma once

#include "common.cuh"

namespace nvfp4_mla {

constexpr int kTile = 128;           // top-k slots per pipeline tile (two 64-slot sub-tiles)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

struct DecodeParams {
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
  float q_lat_mult;   // latent_scale for FP8 rows, else 1 (folded into q)
  float q_rope_mult;  // rope_scale (folded into q)
  float out_mult;     // latent_scale for FP8 rows, else 1
  void* out;
  int32_t out_fp32;
  float* lse;
  float* ws;          // [num_q, splits, H, 512] partial O, then [num_q, splits, H] partial LSE
  int32_t num_splits, tiles_per_split, num_tiles;
  int32_t* invalid_count;
  int32_t use_tma;    // rows gathered with tile::gather4 tensor copies (else one bulk copy per row)
  long long wait_cycles;  // bound of every wait inside the kernel (clock cycles)
};

// Bound of the decode kernel's waits: the default, or the process-wide
// override set through nvfp4_mla_set_wait_limit.
long long decode_wait_cycles();

// Enqueue the tensor-core decode kernel (one 2-CTA cluster per (token, split)).
int32_t launch_decode_tc(const DecodeParams& p, int row_format, cudaStream_t stream);

}  // namespace nvfp4_mla
