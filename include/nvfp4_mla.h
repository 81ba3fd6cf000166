/*
 * nvfp4_mla.h -- C ABI of the NVFP4-compressed MLA KV cache and its sparse
 * decode attention, for NVIDIA GB300 (sm_103a).
 *
 * Source of the method: the Prime Inference post ("Prime Inference: Fast,
 * Reliable Serving for Frontier Open Models"),
 *   section "Making room for low-latency decode"  -- the cache row format;
 *   section "Native NVFP4 sparse MLA decode kernel" -- the fused decode.
 *
 * Conventions shared by every entry point:
 *   - Pointers marked "device" must point to memory of the current CUDA
 *     device; the caller owns all memory. The library allocates nothing and
 *     keeps no per-call state (only a per-device cache of the SM count).
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream). All work is enqueued asynchronously on it; nothing
 *     synchronises the host.
 *   - A nonzero return value is an nvfp4_mla_status. Argument errors are
 *     detected on the host before anything is enqueued. Data errors inside
 *     device buffers (indices, block-table entries) never fault: the
 *     affected entries are skipped and, when `invalid_count` is given,
 *     counted into it with atomicAdd (the caller zeroes it).
 *   - bf16 means IEEE-754 binary16 "brain float" (1-8-7), stored as 16-bit
 *     words; int32 indices are little-endian two's complement.
 *
 * The cache: a pool of `num_blocks` physical pages; page p starts at byte
 * p * block_stride_bytes of `cache` and holds `page_size` rows of
 * row_bytes(row_format) bytes each. A token at logical position `pos` of
 * sequence `s` lives in page block_table[s * max_blocks_per_seq +
 * pos / page_size], row pos % page_size. block_stride_bytes may exceed
 * page_size * row_bytes (e.g. pages that interleave several layers).
 *
 * NVFP4 row (352 bytes, row_format = NVFP4_MLA_ROW_NVFP4_352):
 *   bytes   0..255  E2M1 codes of the 512 latent values, element 2i in the
 *                   low nibble of byte i, element 2i+1 in the high nibble;
 *   bytes 256..287  one E4M3 scale per 16 latent values;
 *   bytes 288..351  the 64 rope values as E4M3.
 * Encoding (this library's reading of the post, which fixes only the
 * format): scale = E4M3(amax/6) (nearest, ties to even, saturating to
 * 448); code = E2M1 nearest to x/scale (ties to the even code, saturating
 * at 6, sign from x; a zero scale gives code 0); rope byte =
 * E4M3(fp32(r / rope_scale)).
 * FP8 row (576 bytes, NVFP4_MLA_ROW_FP8_576), the format the post compares
 * against: 512 bytes E4M3(fp32(x / latent_scale)), then the 64 rope bytes.
 */
#ifndef NVFP4_MLA_H_
#define NVFP4_MLA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define NVFP4_MLA_LATENT_DIM 512
#define NVFP4_MLA_ROPE_DIM 64
#define NVFP4_MLA_SCALE_GROUP 16
#define NVFP4_MLA_NVFP4_ROW_BYTES 352
#define NVFP4_MLA_FP8_ROW_BYTES 576
#define NVFP4_MLA_MAX_HEADS 128
#define NVFP4_MLA_MAX_TOPK 65536

typedef enum nvfp4_mla_status {
  NVFP4_MLA_OK = 0,
  NVFP4_MLA_ERR_NULL = 1,      /* a required pointer is NULL */
  NVFP4_MLA_ERR_SHAPE = 2,     /* a size or count is out of range */
  NVFP4_MLA_ERR_ALIGN = 3,     /* a pointer or stride is not 16-byte aligned */
  NVFP4_MLA_ERR_ARCH = 4,      /* the current device is not sm_103 */
  NVFP4_MLA_ERR_WORKSPACE = 5, /* workspace missing or smaller than required */
  NVFP4_MLA_ERR_LAUNCH = 6,    /* a CUDA call failed while enqueuing */
  NVFP4_MLA_ERR_FORMAT = 7,    /* unknown row_format */
  NVFP4_MLA_ERR_VALUE = 8,     /* a scalar argument is not finite or not positive */
  NVFP4_MLA_ERR_DEVICE = 9     /* no current CUDA device / device query failed */
} nvfp4_mla_status;

typedef enum nvfp4_mla_row_format {
  NVFP4_MLA_ROW_NVFP4_352 = 0,
  NVFP4_MLA_ROW_FP8_576 = 1
} nvfp4_mla_row_format;

/* Bytes of one cache row of `row_format`, or 0 for an unknown format. */
int32_t nvfp4_mla_row_bytes(int32_t row_format);

/* Static description of a status code (never NULL). */
const char* nvfp4_mla_status_string(int32_t status);

/*
 * Quantize-on-append: encode `n_tok` new tokens into their cache rows.
 * Follows the row format of section "Making room for low-latency decode".
 *
 *   latent       device bf16 [n_tok, 512], row-major, 16-byte aligned
 *   rope         device bf16 [n_tok, 64], row-major, 16-byte aligned
 *   seq_ids      device int32 [n_tok]: sequence of each token
 *   positions    device int32 [n_tok]: logical position of each token
 *   block_table  device int32 [num_seqs, max_blocks_per_seq]
 *   cache        device, 16-byte aligned; num_blocks * block_stride_bytes bytes
 *   block_stride_bytes  multiple of 16, >= page_size * row_bytes(row_format)
 *   latent_scale FP8 rows only: latent divisor (finite, > 0; ignored for NVFP4)
 *   rope_scale   rope divisor (finite, > 0)
 *   invalid_count nullable device int32: += tokens whose (sequence, position,
 *                page) does not resolve to a slot; such tokens are not written
 * n_tok = 0 is a no-op returning NVFP4_MLA_OK. Two tokens that resolve to
 * the same slot race (one of them wins). Inputs must be finite.
 */
int32_t nvfp4_mla_append(const void* latent, const void* rope, const int32_t* seq_ids,
                         const int32_t* positions, int32_t n_tok, const int32_t* block_table,
                         int32_t num_seqs, int32_t max_blocks_per_seq, int32_t page_size,
                         void* cache, int64_t num_blocks, int64_t block_stride_bytes,
                         int32_t row_format, float latent_scale, float rope_scale,
                         int32_t* invalid_count, void* stream);

/*
 * Number of top-k splits sparse_mla_decode uses for this shape when its
 * `num_splits` argument is 0 (batch-adaptive, after the post's "adjust the
 * cluster to the batch" change in section "Native NVFP4 sparse MLA decode
 * kernel"). Depends on the SM count of the current device. A split covers
 * at least two 128-slot tiles, and a top-k of fewer than four tiles is not
 * split. Returns >= 1, or 0 when the shape is invalid or the device query
 * fails.
 */
int32_t sparse_mla_decode_num_splits(int32_t num_q, int32_t num_heads, int32_t topk);

/*
 * Workspace bytes sparse_mla_decode needs for this shape and split count
 * (`num_splits` 0 = the automatic choice above). 0 means no workspace is
 * needed (single split). Returns SIZE_MAX for an invalid shape.
 */
size_t sparse_mla_decode_workspace_size(int32_t num_q, int32_t num_heads, int32_t topk,
                                        int32_t num_splits);

/*
 * Sparse absorbed-MLA decode attention over the compressed cache, section
 * "Native NVFP4 sparse MLA decode kernel": the selected rows are gathered
 * at their top-k positions and dequantised on chip (no intermediate FP8
 * buffer in device memory); scores and the weighted sum use FP16 operands
 * with FP32 accumulation; -1 slots are skipped without a load.
 *
 * For query token t (sequence b = q_seq[t]) and head h, over the valid
 * entries j of topk_idx[t]:
 *   z_j = sm_scale * (q_latent[t,h,:] . latent_j + q_rope[t,h,:] . rope_j)
 *   out[t,h,:] = sum_j softmax(z)_j * latent_j      (512 values)
 *   lse[t,h]   = ln(sum_j exp(z_j))                  (natural log)
 * where latent_j / rope_j are the dequantised values of the selected row
 * (rope scaled by rope_scale; FP8 latent scaled by latent_scale). A token
 * with no valid entry gets out = 0 and lse = -inf.
 *
 *   q_latent     device bf16 [num_q, num_heads, 512], 16-byte aligned
 *   q_rope       device bf16 [num_q, num_heads, 64], 16-byte aligned
 *                (|q| must stay below 65504: operands are FP16)
 *   q_seq        device int32 [num_q]
 *   topk_idx     device int32 [num_q, topk]: logical positions; -1 = empty
 *                slot (skipped, not counted); any other entry that does not
 *                resolve (bad q_seq, position < 0 or >= seq_lens[b], page
 *                beyond the table, page id outside [0, num_blocks)) is
 *                skipped and counted into invalid_count
 *   num_heads    1..128; topk 1..65536; num_q >= 0 (0 is a no-op)
 *   block_table  device int32 [num_seqs, max_blocks_per_seq]
 *   seq_lens     device int32 [num_seqs]
 *   cache        device, 16-byte aligned, rows in `row_format`
 *   sm_scale     finite; latent_scale, rope_scale finite and > 0
 *   out          device [num_q, num_heads, 512]: bf16, or fp32 if out_fp32
 *   lse          nullable device fp32 [num_q, num_heads]
 *   workspace    device, 16-byte aligned, >= sparse_mla_decode_workspace_size
 *                bytes for the same shape and num_splits (may be NULL when
 *                that size is 0); scratch, contents need not be initialised
 *   num_splits   0 = automatic; otherwise 1..64, clamped to the number of
 *                128-slot tiles in topk
 *   invalid_count nullable device int32 (accumulated with atomicAdd)
 * Duplicate entries count once each. The result does not depend on the
 * order of entries within a row of topk_idx beyond fp32 rounding.
 */
int32_t sparse_mla_decode(const void* q_latent, const void* q_rope, const int32_t* q_seq,
                          const int32_t* topk_idx, int32_t num_q, int32_t num_heads,
                          int32_t topk, const int32_t* block_table, int32_t num_seqs,
                          int32_t max_blocks_per_seq, const int32_t* seq_lens, int32_t page_size,
                          const void* cache, int64_t num_blocks, int64_t block_stride_bytes,
                          int32_t row_format, float sm_scale, float latent_scale,
                          float rope_scale, void* out, int32_t out_fp32, float* lse,
                          void* workspace, size_t workspace_bytes, int32_t num_splits,
                          int32_t* invalid_count, void* stream);

/*
 * Bound of the decode kernel's internal waits (for gathered rows, for a
 * pipeline slot, for the partner SM of its cluster), in SM clock cycles.
 * A wait that runs out makes its (query token, split) unit give up: the
 * unit drains the copies and tensor-core work it has in flight, frees its
 * tensor memory and writes NaN to its outputs and LSE (or workspace
 * partials), so a stalled launch ends with a visible result instead of
 * holding its SMs. 0 restores the default of 2^31 cycles (about a second).
 * Process-wide; applies to decode launches enqueued after the call. A bound
 * shorter than a healthy launch's waits makes healthy launches fail, which
 * is how the failure path is tested. Returns NVFP4_MLA_ERR_VALUE if
 * cycles < 0. This is this library's choice; the post has no counterpart.
 */
int32_t nvfp4_mla_set_wait_limit(int64_t cycles);

/*
 * sparse_mla_decode without a caller-provided workspace. The paper has no
 * counterpart to this entry point; it exists for callers that cannot
 * allocate device memory themselves -- for example a plugin whose host
 * application owns the device heap through its own allocator and does not
 * let plugins call cudaMalloc, or a service that fixes its device-memory
 * budget at start-up.
 *
 * Arguments, results and errors are those of sparse_mla_decode, minus
 * `workspace` / `workspace_bytes`. When the split-K combine needs scratch
 * (sparse_mla_decode_workspace_size(num_q, num_heads, topk, num_splits) > 0)
 * it uses a static device buffer of NVFP4_MLA_NOALLOC_SCRATCH_BYTES that
 * this library defines; shapes needing more return NVFP4_MLA_ERR_WORKSPACE
 * before anything is enqueued. The entry point allocates nothing and calls
 * no allocating routine.
 *   - The buffer lives in every device that loads the library, until the
 *     process exits (16 MiB each).
 *   - The first call on a device that needs scratch looks up the buffer's
 *     device address (cudaGetSymbolAddress, with that device current) and
 *     caches it; make that first call before any stream capture.
 *   - Every call shares the one buffer: calls whose work can overlap on the
 *     GPU (different streams, or different host threads, without ordering
 *     between them) race on it and corrupt each other's results. Order them
 *     on one stream. Each call fully writes the scratch it reads, so no
 *     clearing is needed between calls.
 */
#define NVFP4_MLA_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)

int32_t sparse_mla_decode_noalloc(const void* q_latent, const void* q_rope, const int32_t* q_seq,
                                  const int32_t* topk_idx, int32_t num_q, int32_t num_heads,
                                  int32_t topk, const int32_t* block_table, int32_t num_seqs,
                                  int32_t max_blocks_per_seq, const int32_t* seq_lens,
                                  int32_t page_size, const void* cache, int64_t num_blocks,
                                  int64_t block_stride_bytes, int32_t row_format, float sm_scale,
                                  float latent_scale, float rope_scale, void* out,
                                  int32_t out_fp32, float* lse, int32_t num_splits,
                                  int32_t* invalid_count, void* stream);

/*
 * Merge attention states computed over disjoint parts of each query token's
 * top-k: the split-K merge of section "Native NVFP4 sparse MLA decode kernel"
 * (there across the SMs of a cluster) for parts computed elsewhere, e.g. by
 * the GPUs of a decode-context-parallel group, each running
 * sparse_mla_decode (out_fp32 = 1) on its share of the top-k.
 *
 *   part_out   device fp32 [num_parts, num_q, num_heads, 512], 16-byte aligned:
 *              each part's normalised output
 *   part_lse   device fp32 [num_parts, num_q, num_heads]: each part's
 *              natural-log LSE; -inf marks a part with no valid entry
 *   num_parts  1..1024; num_heads 1..128; num_q >= 0 (0 is a no-op)
 *   out        device [num_q, num_heads, 512]: bf16, or fp32 if out_fp32
 *   lse        nullable device fp32 [num_q, num_heads]
 * out = sum_p exp(lse_p - lse) * out_p and lse = ln sum_p exp(lse_p); a
 * (token, head) whose parts are all empty gets out = 0 and lse = -inf.
 * Equal to a single sparse_mla_decode over the union of the parts' entries
 * up to fp32 rounding.
 */
int32_t sparse_mla_merge_states(const float* part_out, const float* part_lse, int32_t num_parts,
                                int32_t num_q, int32_t num_heads, void* out, int32_t out_fp32,
                                float* lse, void* stream);

/*
 * The staged-dequant comparison path of section "Native NVFP4 sparse MLA
 * decode kernel": the post measures its fused kernel against a variant that
 * first dequantises the selected rows into an FP8 temporary buffer in device
 * memory and then runs the attention over that buffer. These two entry
 * points build that buffer from an NVFP4 cache, so sparse_mla_decode with
 * row_format NVFP4_MLA_ROW_FP8_576 can be run over it and the two paths
 * timed on the same inputs. Not part of the fused decode.
 *
 * nvfp4_mla_staged_rows_per_q: staged rows per query token, topk rounded up
 * to a multiple of page_size (each token's rows start a page); 0 for an
 * invalid topk (outside 1..65536) or page_size (outside 1..2^20).
 *
 * nvfp4_mla_stage_fp8: for query token t and slot j of topk_idx[t] that
 * resolves as in sparse_mla_decode (same rules, same invalid_count), the
 * NVFP4 row is decoded (E2M1 code x E4M3 block scale, exact in fp32) and
 * re-encoded as an FP8 row: latent byte = E4M3(fp32(value / latent_scale)),
 * nearest with ties to even, saturating to +-448; the 64 rope bytes are
 * copied (both formats store E4M3(rope / rope_scale)). The row is written
 * to staged row t * R + j (R = nvfp4_mla_staged_rows_per_q(topk,
 * page_size)) and staged_idx[t * topk + j] = j; a slot that does not
 * resolve gets staged_idx = -1 and its staged row is left untouched.
 *
 *   q_seq .. block_stride_bytes  as for sparse_mla_decode, with an NVFP4 cache
 *   latent_scale  finite, > 0: the FP8 rows' latent divisor
 *   staged        device, 16-byte aligned, num_q * R * 576 bytes: the
 *                 staged rows, contiguous
 *   staged_idx    device int32 [num_q, topk]
 *   invalid_count nullable device int32 (accumulated with atomicAdd)
 *
 * Reading the staged rows back with sparse_mla_decode: row_format FP8,
 * the same latent_scale and rope_scale, cache = staged, page_size as here,
 * block_stride_bytes = page_size * 576, num_blocks = num_q * R / page_size,
 * num_seqs = num_q, max_blocks_per_seq = R / page_size, q_seq[t] = t,
 * block_table[t][k] = t * (R / page_size) + k, seq_lens[t] = topk,
 * topk_idx = staged_idx.
 */
int64_t nvfp4_mla_staged_rows_per_q(int32_t topk, int32_t page_size);

int32_t nvfp4_mla_stage_fp8(const int32_t* q_seq, const int32_t* topk_idx, int32_t num_q,
                            int32_t topk, const int32_t* block_table, int32_t num_seqs,
                            int32_t max_blocks_per_seq, const int32_t* seq_lens,
                            int32_t page_size, const void* cache, int64_t num_blocks,
                            int64_t block_stride_bytes, float latent_scale, void* staged,
                            int32_t* staged_idx, int32_t* invalid_count, void* stream);

#ifdef __cplusplus
} /* extern "C" */
#endif

#endif /* NVFP4_MLA_H_ */
