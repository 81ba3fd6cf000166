/*
 * nvfp4_mla_oracle.c -- plain, slow CPU oracle for the NVFP4-compressed MLA
 * decode path. TEST INFRASTRUCTURE ONLY: tests, the smoke check and the
 * benchmark's CPU-baseline leg may call it; the product path never does.
 * It shares no code, header, table or constant generator with the CUDA
 * library, and includes nothing from it.
 *
 * What it computes, from the Prime Inference post ("Prime Inference: Fast,
 * Reliable Serving for Frontier Open Models"):
 *   - section "Making room for low-latency decode": the 512-value MLA latent
 *     is stored as NVFP4 (4-bit values, one FP8 scale per 16 values), the
 *     64-value positional (rope) part stays FP8, and a cache row shrinks
 *     from 576 to 352 bytes;
 *   - section "Native NVFP4 sparse MLA decode kernel": attention reads the
 *     compressed rows at the indexer-selected positions, dequantises them,
 *     and computes with FP16 operands / FP32 accumulation; empty slots of
 *     the position list are marked -1 and are not read.
 * Readings where the post is silent (all stated again in the design notes):
 *   - block scale = amax/6 rounded to E4M3 (nearest, ties to even,
 *     saturating at 448); element = x/scale rounded to the E2M1 grid
 *     (nearest, ties to the even code, saturating at 6); a zero scale gives
 *     code 0; the sign bit follows the sign of x (so a negative value that
 *     rounds to 0 is stored as -0);
 *   - two elements per byte, the even-indexed one in the low nibble;
 *   - row = [256 B E2M1 payload][32 B E4M3 scales][64 B E4M3 rope];
 *   - rope byte = E4M3(fp32(r / rope_scale)); the FP8 576-byte comparator
 *     row = [512 B E4M3(fp32(x / latent_scale))][64 B rope];
 *   - absorbed-MLA attention: z = sm_scale * (q_lat . lat + q_rope . rope),
 *     softmax over the valid selected rows, out = sum_j p_j lat_j,
 *     lse = natural-log log-sum-exp of z; no valid row -> out 0, lse -inf;
 *   - an entry other than -1 that does not resolve to a cache row (bad
 *     sequence, position >= seq_len, page beyond the table, physical page
 *     outside the pool) is skipped and counted as invalid.
 * Every floating-point step is fp64 except where a reading fixes fp32 (the
 * rope and FP8-latent quotients). Encoders are brute-force nearest-value
 * searches over every finite code.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_LATENT 512
#define ORC_ROPE 64
#define ORC_BLOCK 16
#define ORC_NVFP4_ROW 352 /* 512/2 + 512/16 + 64 */
#define ORC_FP8_ROW 576   /* 512 + 64 */

/* ---------------------------------------------------------------- bf16 */
double orc_bf16_to_f64(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

static float bf16_to_f32(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

/* ---------------------------------------------------------------- E4M3 */
/* OCP FP8 E4M3 ("FN"): 1 sign, 4 exponent (bias 7), 3 mantissa bits.
 * Exponent field 0 is subnormal (m/8 * 2^-6); S.1111.111 is NaN; there is
 * no infinity, so the largest finite magnitude is 1.75 * 2^8 = 448. */
double orc_e4m3_decode(uint8_t c) {
  int s = c >> 7, e = (c >> 3) & 15, m = c & 7;
  double mag;
  if (e == 15 && m == 7) return NAN;
  if (e == 0)
    mag = ldexp((double)m / 8.0, -6);
  else
    mag = ldexp(1.0 + (double)m / 8.0, e - 7);
  return s ? -mag : mag;
}

/* E2M1 (FP4): 1 sign, 2 exponent (bias 1), 1 mantissa bit. Exponent 0 is
 * subnormal (m * 0.5). Magnitudes: 0, 0.5, 1, 1.5, 2, 3, 4, 6. */
double orc_e2m1_decode(uint8_t c) {
  int s = (c >> 3) & 1, e = (c >> 1) & 3, m = c & 1;
  double mag = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
  return s ? -mag : mag;
}

/* Index of the code in [0, ncodes) whose value is nearest to a >= 0; an
 * exact tie between two neighbours goes to the even code (the one whose
 * mantissa LSB is 0). Searching only finite codes makes values beyond the
 * largest one saturate to it. */
static int nearest_code(double a, double (*dec)(uint8_t), int ncodes) {
  int best = 0;
  double bd = fabs(a - dec(0));
  for (int c = 1; c < ncodes; ++c) {
    double d = fabs(a - dec((uint8_t)c));
    if (d < bd || (d == bd && (c & 1) == 0 && (best & 1) == 1)) {
      best = c;
      bd = d;
    }
  }
  return best;
}

/* Round x to E4M3: nearest finite value, ties to even, saturating at
 * +-448; the sign bit copies the sign of x (also for results of 0).
 * Magnitudes >= 448 saturate before the search: far above the range the
 * fp64 distances to the top codes round to the same value. */
uint8_t orc_e4m3_encode(double x) {
  int mag = fabs(x) >= 448.0 ? 0x7E : nearest_code(fabs(x), orc_e4m3_decode, 0x7F);
  return (uint8_t)((signbit(x) ? 0x80 : 0x00) | mag);
}

/* Round v to E2M1: nearest grid value, ties to the even code, saturating
 * at +-6; the sign bit copies the sign of v. */
uint8_t orc_e2m1_encode(double v) {
  int mag = fabs(v) >= 6.0 ? 7 : nearest_code(fabs(v), orc_e2m1_decode, 8);
  return (uint8_t)((signbit(v) ? 0x8 : 0x0) | mag);
}

/* ----------------------------------------------------------- row codec */
/* One NVFP4 cache row from bf16 latent[512] and rope[64]. */
void orc_quantize_row_nvfp4(const uint16_t* lat, const uint16_t* rope, float rope_scale,
                            uint8_t* row) {
  uint8_t codes[ORC_LATENT];
  for (int j = 0; j < ORC_LATENT / ORC_BLOCK; ++j) {
    double amax = 0.0;
    for (int k = 0; k < ORC_BLOCK; ++k) amax = fmax(amax, fabs(orc_bf16_to_f64(lat[ORC_BLOCK * j + k])));
    uint8_t sc = orc_e4m3_encode(amax / 6.0);
    double S = orc_e4m3_decode(sc);
    row[256 + j] = sc;
    for (int k = 0; k < ORC_BLOCK; ++k) {
      double x = orc_bf16_to_f64(lat[ORC_BLOCK * j + k]);
      codes[ORC_BLOCK * j + k] = (S == 0.0) ? 0 : orc_e2m1_encode(x / S);
    }
  }
  for (int i = 0; i < ORC_LATENT / 2; ++i)
    row[i] = (uint8_t)(codes[2 * i] | (codes[2 * i + 1] << 4));
  for (int k = 0; k < ORC_ROPE; ++k) {
    float q = bf16_to_f32(rope[k]) / rope_scale; /* fp32 quotient, IEEE rounded */
    row[288 + k] = orc_e4m3_encode((double)q);
  }
}

/* One FP8 (576-byte) comparator row. */
void orc_quantize_row_fp8(const uint16_t* lat, const uint16_t* rope, float latent_scale,
                          float rope_scale, uint8_t* row) {
  for (int k = 0; k < ORC_LATENT; ++k) {
    float q = bf16_to_f32(lat[k]) / latent_scale;
    row[k] = orc_e4m3_encode((double)q);
  }
  for (int k = 0; k < ORC_ROPE; ++k) {
    float q = bf16_to_f32(rope[k]) / rope_scale;
    row[ORC_LATENT + k] = orc_e4m3_encode((double)q);
  }
}

/* Decoded values of one row (fp64, exact). */
void orc_dequant_row(const uint8_t* row, int row_format, float latent_scale, float rope_scale,
                     double* lat, double* rope) {
  if (row_format == 0) {
    for (int k = 0; k < ORC_LATENT; ++k) {
      uint8_t b = row[k / 2];
      uint8_t code = (k & 1) ? (b >> 4) : (b & 15);
      lat[k] = orc_e2m1_decode(code) * orc_e4m3_decode(row[256 + k / ORC_BLOCK]);
    }
    for (int k = 0; k < ORC_ROPE; ++k) rope[k] = orc_e4m3_decode(row[288 + k]) * (double)rope_scale;
  } else {
    for (int k = 0; k < ORC_LATENT; ++k) lat[k] = orc_e4m3_decode(row[k]) * (double)latent_scale;
    for (int k = 0; k < ORC_ROPE; ++k) rope[k] = orc_e4m3_decode(row[ORC_LATENT + k]) * (double)rope_scale;
  }
}

int orc_row_bytes(int row_format) { return row_format == 0 ? ORC_NVFP4_ROW : ORC_FP8_ROW; }

/* ------------------------------------------------------- paged address */
/* Byte offset of (seq, pos) in the pool, or -1 when it does not resolve:
 * page = block_table[seq][pos / page_size], row = pos % page_size. */
static int64_t resolve(int32_t seq, int32_t pos, int32_t seq_len_or_neg, const int32_t* block_table,
                       int32_t num_seqs, int32_t max_blocks, int32_t page_size, int64_t num_blocks,
                       int64_t block_stride, int row_bytes) {
  if (seq < 0 || seq >= num_seqs || pos < 0) return -1;
  if (seq_len_or_neg >= 0 && pos >= seq_len_or_neg) return -1;
  int64_t lb = pos / page_size;
  if (lb >= max_blocks) return -1;
  int64_t pb = block_table[(int64_t)seq * max_blocks + lb];
  if (pb < 0 || pb >= num_blocks) return -1;
  return pb * block_stride + (int64_t)(pos % page_size) * row_bytes;
}

/* Quantize-on-append: encode each token's row and store it at its paged
 * slot. Tokens that do not resolve are skipped; returns how many. */
int64_t orc_append(const uint16_t* latent, const uint16_t* rope, const int32_t* seq_ids,
                   const int32_t* positions, int32_t n_tok, const int32_t* block_table,
                   int32_t num_seqs, int32_t max_blocks, int32_t page_size, uint8_t* cache,
                   int64_t num_blocks, int64_t block_stride, int32_t row_format,
                   float latent_scale, float rope_scale) {
  int rb = orc_row_bytes(row_format);
  int64_t bad = 0;
  for (int32_t t = 0; t < n_tok; ++t) {
    int64_t off = resolve(seq_ids[t], positions[t], -1, block_table, num_seqs, max_blocks,
                          page_size, num_blocks, block_stride, rb);
    if (off < 0) { ++bad; continue; }
    const uint16_t* l = latent + (int64_t)t * ORC_LATENT;
    const uint16_t* r = rope + (int64_t)t * ORC_ROPE;
    if (row_format == 0)
      orc_quantize_row_nvfp4(l, r, rope_scale, cache + off);
    else
      orc_quantize_row_fp8(l, r, latent_scale, rope_scale, cache + off);
  }
  return bad;
}

/* ------------------------------------------------------------ attention */
/* Sparse absorbed-MLA decode. For query token t (sequence q_seq[t]) and
 * head h, over the valid entries j of topk_idx[t]:
 *   z_j = sm_scale * (sum_512 q_lat * lat_j + sum_64 q_rope * rope_j)
 *   out[t,h,:] = sum_j softmax(z)_j * lat_j,  lse[t,h] = log sum_j exp(z_j)
 * out is [num_q, H, 512] fp64, lse [num_q, H] fp64. Returns the number of
 * entries that are neither -1 nor a resolvable row. nthreads <= 0 uses the
 * OpenMP default; the parallel loop is over heads of one query token. */
int64_t orc_sparse_mla_decode(const uint16_t* q_lat, const uint16_t* q_rope, const int32_t* q_seq,
                              const int32_t* topk_idx, int32_t num_q, int32_t num_heads,
                              int32_t topk, const int32_t* block_table, int32_t num_seqs,
                              int32_t max_blocks, const int32_t* seq_lens, int32_t page_size,
                              const uint8_t* cache, int64_t num_blocks, int64_t block_stride,
                              int32_t row_format, float sm_scale, float latent_scale,
                              float rope_scale, double* out, double* lse, int nthreads) {
  int rb = orc_row_bytes(row_format);
  int64_t bad = 0;
  double* lat = (double*)malloc(sizeof(double) * (size_t)(topk > 0 ? topk : 1) * ORC_LATENT);
  double* rp = (double*)malloc(sizeof(double) * (size_t)(topk > 0 ? topk : 1) * ORC_ROPE);
  for (int32_t t = 0; t < num_q; ++t) {
    int32_t b = q_seq[t];
    int n = 0;
    for (int32_t j = 0; j < topk; ++j) {
      int32_t pos = topk_idx[(int64_t)t * topk + j];
      if (pos == -1) continue;
      int32_t len = (b >= 0 && b < num_seqs) ? seq_lens[b] : 0;
      int64_t off = resolve(b, pos, len, block_table, num_seqs, max_blocks, page_size,
                            num_blocks, block_stride, rb);
      if (off < 0) { ++bad; continue; }
      orc_dequant_row(cache + off, row_format, latent_scale, rope_scale,
                      lat + (int64_t)n * ORC_LATENT, rp + (int64_t)n * ORC_ROPE);
      ++n;
    }
    int nt = nthreads;
#ifdef _OPENMP
    if (nt <= 0) nt = omp_get_max_threads();
#pragma omp parallel for num_threads(nt) schedule(static)
#endif
    for (int32_t h = 0; h < num_heads; ++h) {
      const uint16_t* ql = q_lat + ((int64_t)t * num_heads + h) * ORC_LATENT;
      const uint16_t* qr = q_rope + ((int64_t)t * num_heads + h) * ORC_ROPE;
      double* o = out + ((int64_t)t * num_heads + h) * ORC_LATENT;
      double* z = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
      double m = -INFINITY;
      for (int i = 0; i < n; ++i) {
        double s = 0.0;
        for (int k = 0; k < ORC_LATENT; ++k) s += orc_bf16_to_f64(ql[k]) * lat[(int64_t)i * ORC_LATENT + k];
        for (int k = 0; k < ORC_ROPE; ++k) s += orc_bf16_to_f64(qr[k]) * rp[(int64_t)i * ORC_ROPE + k];
        z[i] = (double)sm_scale * s;
        if (z[i] > m) m = z[i];
      }
      for (int k = 0; k < ORC_LATENT; ++k) o[k] = 0.0;
      if (n == 0) {
        lse[(int64_t)t * num_heads + h] = -INFINITY;
      } else {
        double Z = 0.0;
        for (int i = 0; i < n; ++i) Z += exp(z[i] - m);
        for (int i = 0; i < n; ++i) {
          double p = exp(z[i] - m) / Z;
          for (int k = 0; k < ORC_LATENT; ++k) o[k] += p * lat[(int64_t)i * ORC_LATENT + k];
        }
        lse[(int64_t)t * num_heads + h] = m + log(Z);
      }
      free(z);
    }
  }
  free(lat);
  free(rp);
  return bad;
}

/* Staged-dequant comparison path (section "Native NVFP4 sparse MLA decode
 * kernel": the post times its fused kernel against dequantising the selected
 * rows into an FP8 temporary buffer first). For query token t and slot j
 * that resolves in an NVFP4 cache, the row's latent values (code x block
 * scale, exact) are re-encoded as E4M3 of the fp32 quotient value /
 * latent_scale (nearest, ties to even, saturating), the rope bytes copied,
 * and the 576-byte row stored as staged row t * rows_per_q + j with
 * staged_idx = j. Slots that do not resolve get staged_idx = -1; those
 * other than -1 are counted (returned). */
int64_t orc_stage_fp8(const int32_t* q_seq, const int32_t* topk_idx, int32_t num_q, int32_t topk,
                      const int32_t* block_table, int32_t num_seqs, int32_t max_blocks,
                      const int32_t* seq_lens, int32_t page_size, const uint8_t* cache,
                      int64_t num_blocks, int64_t block_stride, float latent_scale,
                      int64_t rows_per_q, uint8_t* staged, int32_t* staged_idx) {
  int64_t bad = 0;
  double lat[ORC_LATENT], rope[ORC_ROPE];
  for (int32_t t = 0; t < num_q; ++t) {
    int32_t b = q_seq[t];
    int32_t len = (b >= 0 && b < num_seqs) ? seq_lens[b] : 0;
    for (int32_t j = 0; j < topk; ++j) {
      int32_t pos = topk_idx[(int64_t)t * topk + j];
      int64_t off = pos == -1 ? -1
                              : resolve(b, pos, len, block_table, num_seqs, max_blocks, page_size,
                                        num_blocks, block_stride, ORC_NVFP4_ROW);
      staged_idx[(int64_t)t * topk + j] = off >= 0 ? j : -1;
      if (off < 0) {
        if (pos != -1) ++bad;
        continue;
      }
      const uint8_t* row = cache + off;
      uint8_t* dst = staged + ((int64_t)t * rows_per_q + j) * ORC_FP8_ROW;
      orc_dequant_row(row, 0, 1.0f, 1.0f, lat, rope);
      for (int k = 0; k < ORC_LATENT; ++k) {
        float q = (float)lat[k] / latent_scale; /* value exact in fp32; quotient IEEE rounded */
        dst[k] = orc_e4m3_encode((double)q);
      }
      for (int k = 0; k < ORC_ROPE; ++k) dst[ORC_LATENT + k] = row[288 + k];
    }
  }
  return bad;
}

/* Merge of attention states over disjoint parts of each query token's
 * selection (section "Native NVFP4 sparse MLA decode kernel": a token's
 * partial softmax results are merged; here parts from anywhere). Each part
 * is a normalised output out_p [512] with its natural-log lse_p; with
 * m = max_p lse_p: out = sum_p exp(lse_p - m) out_p / sum_p exp(lse_p - m),
 * lse = m + ln sum_p exp(lse_p - m). All parts empty (-inf) -> 0, -inf.
 * Layout: part_out [P][states][512], part_lse [P][states]. */
void orc_merge_states(const double* part_out, const double* part_lse, int32_t num_parts,
                      int64_t states, double* out, double* lse) {
  for (int64_t i = 0; i < states; ++i) {
    double m = -INFINITY;
    for (int p = 0; p < num_parts; ++p)
      if (part_lse[p * states + i] > m) m = part_lse[p * states + i];
    double* o = out + i * ORC_LATENT;
    for (int k = 0; k < ORC_LATENT; ++k) o[k] = 0.0;
    if (m == -INFINITY) {
      lse[i] = -INFINITY;
      continue;
    }
    double tot = 0.0;
    for (int p = 0; p < num_parts; ++p) {
      double w = exp(part_lse[p * states + i] - m);
      tot += w;
      for (int k = 0; k < ORC_LATENT; ++k) o[k] += w * part_out[(p * states + i) * ORC_LATENT + k];
    }
    for (int k = 0; k < ORC_LATENT; ++k) o[k] /= tot;
    lse[i] = m + log(tot);
  }
}

int orc_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* ------------------------------------------------ array entry points */
void orc_e4m3_encode_n(const double* x, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_e4m3_encode(x[i]);
}
void orc_e4m3_decode_n(const uint8_t* c, int64_t n, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_e4m3_decode(c[i]);
}
void orc_e2m1_encode_n(const double* v, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_e2m1_encode(v[i]);
}
void orc_e2m1_decode_n(const uint8_t* c, int64_t n, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_e2m1_decode(c[i]);
}
void orc_quantize_rows(const uint16_t* lat, const uint16_t* rope, int64_t n, int32_t row_format,
                       float latent_scale, float rope_scale, uint8_t* rows) {
  int rb = orc_row_bytes(row_format);
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
  for (int64_t i = 0; i < n; ++i) {
    if (row_format == 0)
      orc_quantize_row_nvfp4(lat + i * ORC_LATENT, rope + i * ORC_ROPE, rope_scale, rows + i * rb);
    else
      orc_quantize_row_fp8(lat + i * ORC_LATENT, rope + i * ORC_ROPE, latent_scale, rope_scale,
                           rows + i * rb);
  }
}
void orc_dequant_rows(const uint8_t* rows, int64_t n, int32_t row_format, float latent_scale,
                      float rope_scale, double* lat, double* rope) {
  int rb = orc_row_bytes(row_format);
  for (int64_t i = 0; i < n; ++i)
    orc_dequant_row(rows + i * rb, row_format, latent_scale, rope_scale, lat + i * ORC_LATENT,
                    rope + i * ORC_ROPE);
}
