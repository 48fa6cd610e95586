/*
 * Plain CPU oracle for sparse MLA decode attention over a paged FP8 KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or calls this
 * file: only the tests, the package smoke check and the benchmark's CPU-baseline leg
 * do.  It shares no code, header, table or constant with the CUDA library.
 *
 * Everything here is fp64, written as the plain definition, with no blocking, no online
 * softmax and no reordering beyond what the definition states.
 *
 * Sources (page titles and sections):
 *  - "FlashMLA 与 DSA：内核、流水线和正确性边界", section 4.3 (Stage 3 - Sparse Attention):
 *    the semantic definition: gather the selected rows, S = q . K^T * sm_scale, invalid
 *    slots get -inf, lse = logsumexp(S), O = exp(S - lse) . V with V = the first 512
 *    dims of the same rows.
 *  - same page, section 3.1 and "FlashMLA Sparse Decode 完整计算过程详解", steps 2.2 and
 *    4.3: the 656-byte row = 512 e4m3 NoPE codes, 4 little-endian fp32 scales (one per
 *    128-dim group, stored as the dequant multiplier), 64 bf16 RoPE values.
 *  - "FlashMLA Sparse Decode 完整计算过程详解", step 1 and step 7.2: an index is a
 *    physical token id = page * page_block_size + offset; -1 marks an invalid slot.
 *  - same page, step 14.2: a row with no valid slot yields lse = +inf; its output is
 *    defined here as 0.
 *
 * E4M3 is decoded from its integer fields (OCP 8-bit floating point, E4M3 variant):
 * sign s, 4-bit exponent E with bias 7, 3-bit mantissa M; E >= 1 gives
 * (-1)^s 2^(E-7) (1 + M/8); E = 0 gives (-1)^s 2^-6 (M/8); E = 15, M = 7 is NaN.
 * bf16 is decoded from its fields (1 sign, 8 exponent bits with bias 127, 7 mantissa
 * bits), fp32 scales from their little-endian IEEE binary32 bytes.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_D_NOPE 512
#define ORACLE_D_ROPE 64
#define ORACLE_D_QK 576
#define ORACLE_D_V 512
#define ORACLE_ROW_BYTES 656
#define ORACLE_GROUP 128

double smla_oracle_e4m3(uint8_t code) {
  int s = (code >> 7) & 1;
  int e = (code >> 3) & 0xF;
  int m = code & 0x7;
  double mag;
  if (e == 15 && m == 7) return NAN;
  if (e == 0)
    mag = ldexp((double)m / 8.0, -6);
  else
    mag = ldexp(1.0 + (double)m / 8.0, e - 7);
  return s ? -mag : mag;
}

double smla_oracle_bf16(uint16_t bits) {
  int s = (bits >> 15) & 1;
  int e = (bits >> 7) & 0xFF;
  int m = bits & 0x7F;
  double mag;
  if (e == 255) return m ? NAN : (s ? -INFINITY : INFINITY);
  if (e == 0)
    mag = ldexp((double)m / 128.0, -126);
  else
    mag = ldexp(1.0 + (double)m / 128.0, e - 127);
  return s ? -mag : mag;
}

static double oracle_f32_le(const uint8_t* p) {
  uint32_t u = (uint32_t)p[0] | ((uint32_t)p[1] << 8) | ((uint32_t)p[2] << 16) |
               ((uint32_t)p[3] << 24);
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

static uint16_t oracle_u16_le(const uint8_t* p) {
  return (uint16_t)((uint16_t)p[0] | ((uint16_t)p[1] << 8));
}

/* Decode the 576 key dims of one 656-byte row: K[d] = e4m3(byte d) * scale[d / 128] for
 * d < 512 (the product taken exactly in fp64), K[512 + i] = bf16 RoPE value i. */
void smla_oracle_decode_row(const uint8_t* row, double* k) {
  for (int d = 0; d < ORACLE_D_NOPE; ++d) {
    double scale = oracle_f32_le(row + ORACLE_D_NOPE + 4 * (d / ORACLE_GROUP));
    k[d] = smla_oracle_e4m3(row[d]) * scale;
  }
  for (int i = 0; i < ORACLE_D_ROPE; ++i)
    k[ORACLE_D_NOPE + i] = smla_oracle_bf16(oracle_u16_le(row + ORACLE_D_NOPE + 16 + 2 * i));
}

void smla_oracle_e4m3_array(const uint8_t* codes, double* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = smla_oracle_e4m3(codes[i]);
}

void smla_oracle_bf16_array(const uint16_t* bits, double* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = smla_oracle_bf16(bits[i]);
}

/*
 * Sparse MLA decode for a list of query tokens.
 *
 *   q        bf16 bits, [b, s_q, h_q, 576] row-major
 *   kv       bytes, [num_blocks, page_block_size, 656] row-major (h_kv = 1)
 *   indices  int32, [b, s_q, topk]; a slot is valid iff 0 <= idx < num_blocks*page_block_size
 *   tokens   flattened query-token ids (bi * s_q + si) to compute; n_tokens of them
 *   slot_begin, slot_end   only slots in [slot_begin, slot_end) take part (the whole list
 *            is [0, topk)); a sub-range gives the partial result of one split
 *   out      fp64 [n_tokens, h_q, 512]
 *   lse      fp64 [n_tokens, h_q], natural log
 *   n_valid  int32 [n_tokens] (may be NULL): number of valid slots seen
 *
 * Returns 0, or -1 on an allocation failure.
 */
int smla_oracle_sparse_decode(int b, int s_q, int h_q, int topk, int64_t num_blocks,
                              int page_block_size, const uint16_t* q, const uint8_t* kv,
                              const int32_t* indices, double sm_scale, const int32_t* tokens,
                              int n_tokens, int slot_begin, int slot_end, double* out,
                              double* lse, int32_t* n_valid, int num_threads) {
  (void)b;
  int64_t num_slots_pool = num_blocks * (int64_t)page_block_size;
  if (slot_begin < 0) slot_begin = 0;
  if (slot_end > topk) slot_end = topk;
  int max_rows = slot_end > slot_begin ? slot_end - slot_begin : 0;
  double* kbuf = (double*)malloc(sizeof(double) * (size_t)(max_rows > 0 ? max_rows : 1) * ORACLE_D_QK);
  int32_t* rows = (int32_t*)malloc(sizeof(int32_t) * (size_t)(max_rows > 0 ? max_rows : 1));
  if (!kbuf || !rows) {
    free(kbuf);
    free(rows);
    return -1;
  }
#ifdef _OPENMP
  if (num_threads > 0) omp_set_num_threads(num_threads);
#else
  (void)num_threads;
#endif
  for (int t = 0; t < n_tokens; ++t) {
    int tok = tokens[t];
    const int32_t* idx = indices + (int64_t)tok * topk;
    /* Step 1: the ordered list of valid slots, duplicates kept. */
    int n = 0;
    for (int j = slot_begin; j < slot_end; ++j) {
      int64_t id = idx[j];
      if (id >= 0 && id < num_slots_pool) rows[n++] = (int32_t)id;
    }
    if (n_valid) n_valid[t] = n;
    /* Step 2: decode each selected row; page = id / page_block_size, offset = id % page_block_size. */
#pragma omp parallel for schedule(static)
    for (int r = 0; r < n; ++r) {
      int64_t id = rows[r];
      int64_t page = id / page_block_size;
      int64_t off = id % page_block_size;
      const uint8_t* row = kv + (page * page_block_size + off) * ORACLE_ROW_BYTES;
      smla_oracle_decode_row(row, kbuf + (int64_t)r * ORACLE_D_QK);
    }
    /* Step 3: per head, scores, log-sum-exp and the weighted sum of V = K[:, :512]. */
#pragma omp parallel for schedule(dynamic, 1)
    for (int h = 0; h < h_q; ++h) {
      const uint16_t* qh = q + ((int64_t)tok * h_q + h) * ORACLE_D_QK;
      double qd[ORACLE_D_QK];
      double* o = out + ((int64_t)t * h_q + h) * ORACLE_D_V;
      for (int d = 0; d < ORACLE_D_QK; ++d) qd[d] = smla_oracle_bf16(qh[d]);
      for (int d = 0; d < ORACLE_D_V; ++d) o[d] = 0.0;
      if (n == 0) {
        lse[(int64_t)t * h_q + h] = INFINITY;
        continue;
      }
      double* s = (double*)malloc(sizeof(double) * (size_t)n);
      double m = -INFINITY;
      for (int r = 0; r < n; ++r) {
        const double* k = kbuf + (int64_t)r * ORACLE_D_QK;
        double acc = 0.0;
        for (int d = 0; d < ORACLE_D_QK; ++d) acc += qd[d] * k[d];
        s[r] = acc * sm_scale;
        if (s[r] > m) m = s[r];
      }
      double sum = 0.0;
      for (int r = 0; r < n; ++r) sum += exp(s[r] - m);
      double l = m + log(sum);
      lse[(int64_t)t * h_q + h] = l;
      for (int r = 0; r < n; ++r) {
        double p = exp(s[r] - l);
        const double* k = kbuf + (int64_t)r * ORACLE_D_QK;
        for (int d = 0; d < ORACLE_D_V; ++d) o[d] += p * k[d];
      }
      free(s);
    }
  }
  free(kbuf);
  free(rows);
  return 0;
}

int smla_oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
