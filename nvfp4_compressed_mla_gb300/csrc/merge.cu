// merge.cu -- merge of attention states computed over disjoint parts of each
// query token's top-k, for parts that come from outside one decode launch
// (other GPUs of a decode-context-parallel group).
//
// The Prime Inference post, section "Native NVFP4 sparse MLA decode kernel",
// merges a query token's partial softmax results across the SMs of a
// cluster and notes that splitting one token's context over GPUs did not pay
// at 2048 selected tokens. This is the same merge over parts that were
// computed elsewhere: each part is a normalised output with its natural-log
// LSE, exactly what sparse_mla_decode returns for its share of the top-k.
//   out = sum_p exp(lse_p - lse) * out_p,   lse = ln sum_p exp(lse_p)
// HBM-bound: per (token, head) num_parts x (2 KB + 4 B) read, 1-2 KB written.
#include <math.h>

#include "decode_common.cuh"

namespace nvfp4_mla {
namespace {

// One block of 128 threads per (query token, head); thread i owns dims 4i .. 4i + 3.
__global__ void __launch_bounds__(128)
    merge_states_kernel(const float* __restrict__ part_out, const float* __restrict__ part_lse,
                        int32_t num_parts, int64_t states, void* out, int32_t out_fp32,
                        float* lse) {
  const int64_t qh = blockIdx.x;  // t * H + h
  float m = -INFINITY;
  for (int p = 0; p < num_parts; ++p) m = fmaxf(m, __ldg(part_lse + p * states + qh));
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  float tot = 0.f;
  if (m != -INFINITY) {
    for (int p = 0; p < num_parts; ++p) {
      const float w = ex2((__ldg(part_lse + p * states + qh) - m) * kLog2e);  // 0 if empty
      tot += w;
      if (w > 0.f) {
        const float4 v = __ldg(reinterpret_cast<const float4*>(
            part_out + (p * states + qh) * kLatent + threadIdx.x * 4));
        acc[0] += w * v.x;
        acc[1] += w * v.y;
        acc[2] += w * v.z;
        acc[3] += w * v.w;
      }
    }
  }
  const float sc = tot > 0.f ? 1.f / tot : 0.f;
  const int d = threadIdx.x * 4;
  if (out_fp32) {
    *reinterpret_cast<float4*>(static_cast<float*>(out) + qh * kLatent + d) =
        make_float4(acc[0] * sc, acc[1] * sc, acc[2] * sc, acc[3] * sc);
  } else {
    *reinterpret_cast<uint2*>(static_cast<uint16_t*>(out) + qh * kLatent + d) =
        make_uint2(pack_bf16x2(acc[0] * sc, acc[1] * sc), pack_bf16x2(acc[2] * sc, acc[3] * sc));
  }
  if (threadIdx.x == 0 && lse != nullptr) lse[qh] = tot > 0.f ? m + lg2(tot) * kLn2 : -INFINITY;
}

}  // namespace
}  // namespace nvfp4_mla

using namespace nvfp4_mla;

extern "C" int32_t sparse_mla_merge_states(const float* part_out, const float* part_lse,
                                           int32_t num_parts, int32_t num_q, int32_t num_heads,
                                           void* out, int32_t out_fp32, float* lse,
                                           void* stream) {
  if (num_parts < 1 || num_parts > 1024 || num_q < 0 || num_heads < 1 ||
      num_heads > NVFP4_MLA_MAX_HEADS)
    return NVFP4_MLA_ERR_SHAPE;
  if (num_q == 0) return NVFP4_MLA_OK;
  if (!part_out || !part_lse || !out) return NVFP4_MLA_ERR_NULL;
  if (!aligned16(part_out) || !aligned16(out)) return NVFP4_MLA_ERR_ALIGN;
  int dev = 0, sms = 0;
  if (int32_t st = current_device_checked(&dev, &sms)) return st;
  const int64_t states = static_cast<int64_t>(num_q) * num_heads;
  if (states > 0x7FFFFFFF) return NVFP4_MLA_ERR_SHAPE;
  merge_states_kernel<<<static_cast<unsigned>(states), 128, 0,
                        static_cast<cudaStream_t>(stream)>>>(part_out, part_lse, num_parts, states,
                                                             out, out_fp32, lse);
  return launch_status();
}
