/*
 * np_oracle.c -- plain, slow CPU oracle for the batched paged-attention
 * decode read and its KV append.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE.  This file is the reference the CUDA
 * path is checked against.  Only the test suite, the package entry's smoke()
 * and bench.py's CPU-baseline leg load it.  The product library never links,
 * includes or calls it, and the two share no code, header or constant.
 *
 * What it computes, in the pages' terms:
 *
 *  - The cache holds K and V in a pool of fixed-size blocks, and a block table
 *    maps each sequence's logical blocks to physical ones ("Day 17: paging
 *    under the sampling path", Post angle and Diagram).  The pool is read here
 *    as two arrays (one for K, one for V) of shape
 *    [num_blocks, block_size, kv_heads, head_dim], so token t of row r lives
 *    at physical block block_tables[r][t / block_size], offset
 *    t % block_size.
 *
 *  - The read is the same scaled-dot-product attention over the assembled
 *    slots that the torch reference (exact to the byte) computes: gather the row's
 *    whole history by block table, then an exact (two-pass) softmax by index
 *    ("Day 25: the fused read dispatches to the kernel backend", What I added
 *    today and What I learned 1).  One query token per row; it is the newest
 *    position, so every one of the row's context_lens[r] history tokens is
 *    visible (the causal mask removes nothing).
 *
 *  - Query heads share KV heads in groups (GQA, the gqa_attention the read
 *    returns into, same page, Diagram): q head h reads kv head
 *    h / (q_heads / kv_heads).
 *
 *  - A decode step first writes the new token's K/V into its slot,
 *    slot = block * block_size + offset, through a slot mapping ("Day 25",
 *    What I added today: the read receives a slot mapping that covers every
 *    history token); scatter and gather are exact copies (What I learned 1).
 *    A negative slot means "no token" and is skipped.
 *
 *  - For long contexts the history of a (row, head) can be cut into
 *    consecutive token ranges ("splits"); each range yields its own
 *    normalised output and natural-log log-sum-exp, and the full result is the
 *    lse-weighted average of the ranges.  The pages do not describe this
 *    split; it is the flash-decoding partition, and the functions below give
 *    its plain definition so the partials and the combine can be checked on
 *    their own.
 *
 * Arithmetic: every element is widened to the working type (bf16 -> fp32 is
 * exact, fp32 -> fp64 is exact) and scores, softmax and the weighted sum are
 * computed in that type with libm exp/log.  The fp64 instantiation is the
 * primary oracle; the fp32 one follows the pages' own "fp32 softmax" and is
 * used to show that the two agree far inside the kernel tolerance.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { NPO_F32 = 0, NPO_BF16 = 1 };

/* Return codes. */
enum {
  NPO_OK = 0,
  NPO_BAD_ARG = 1,      /* a shape or dtype is not valid */
  NPO_BAD_BLOCK = 2,    /* a block id the walk needs is outside the pool */
  NPO_BAD_CONTEXT = 3,  /* context_lens[r] is negative or above the table */
  NPO_NO_MEMORY = 4
};

/* bf16 is the upper half of an IEEE fp32: widening is a 16-bit shift. */
static float npo_bf16_to_float(uint16_t h) {
  uint32_t bits = (uint32_t)h << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return f;
}

/* Element idx of an array of the given storage type, widened to double. */
static double npo_load(const void* base, int dtype, int64_t idx) {
  if (dtype == NPO_F32) return (double)((const float*)base)[idx];
  return (double)npo_bf16_to_float(((const uint16_t*)base)[idx]);
}

static int npo_elem_size(int dtype) {
  if (dtype == NPO_F32) return 4;
  if (dtype == NPO_BF16) return 2;
  return 0;
}

/* Exported so tests can check the widening against a library conversion. */
double npo_widen(const void* base, int dtype, int64_t idx) {
  return npo_load(base, dtype, idx);
}

/*
 * KV append: for each new token i with slot s = slot_mapping[i] >= 0, copy
 * its [kv_heads, head_dim] K row and V row into pool slot s, byte for byte.
 * Returns NPO_OK, or NPO_BAD_BLOCK when some slot is >= num_blocks *
 * block_size (those tokens are skipped, the others are still written).
 */
int npo_kv_append(void* k_pool, void* v_pool, int dtype, int64_t num_blocks,
                  int32_t block_size, int32_t kv_heads, int32_t head_dim,
                  const void* k_new, const void* v_new,
                  const int64_t* slot_mapping, int32_t num_tokens) {
  int es = npo_elem_size(dtype);
  if (es == 0 || num_blocks <= 0 || block_size <= 0 || kv_heads <= 0 ||
      head_dim <= 0 || num_tokens < 0)
    return NPO_BAD_ARG;
  int64_t row_bytes = (int64_t)kv_heads * head_dim * es;
  int64_t num_slots = num_blocks * block_size;
  int status = NPO_OK;
  for (int32_t i = 0; i < num_tokens; ++i) {
    int64_t s = slot_mapping[i];
    if (s < 0) continue;
    if (s >= num_slots) {
      status = NPO_BAD_BLOCK;
      continue;
    }
    memcpy((char*)k_pool + s * row_bytes, (const char*)k_new + i * row_bytes,
           (size_t)row_bytes);
    memcpy((char*)v_pool + s * row_bytes, (const char*)v_new + i * row_bytes,
           (size_t)row_bytes);
  }
  return status;
}

/* The decode read, once per working precision (see decode_body.h). */
#define NPO_REAL double
#define NPO_EXP exp
#define NPO_LOG log
#define NPO_NAME(x) x##_f64
#include "decode_body.h"
#undef NPO_REAL
#undef NPO_EXP
#undef NPO_LOG
#undef NPO_NAME

#define NPO_REAL float
#define NPO_EXP expf
#define NPO_LOG logf
#define NPO_NAME(x) x##_f32
#include "decode_body.h"
#undef NPO_REAL
#undef NPO_EXP
#undef NPO_LOG
#undef NPO_NAME

/*
 * Combine of split partials (plain definition of the log-sum-exp merge):
 * for each (row, head), with L = max_s lse[s] over the splits,
 *   out = sum_s exp(lse[s] - L) * o[s]  /  sum_s exp(lse[s] - L).
 * Splits with lse = -inf hold no tokens and get weight 0 (their o is not
 * read).  If every split is empty the output is all zeros.
 * o_part: [rows, q_heads, num_splits, head_dim]; lse_part: [rows, q_heads,
 * num_splits]; out: [rows, q_heads, head_dim]; all fp64.
 */
int npo_reduce_f64(double* out, const double* o_part, const double* lse_part,
                   int32_t rows, int32_t q_heads, int32_t num_splits,
                   int32_t head_dim) {
  if (rows < 0 || q_heads <= 0 || num_splits <= 0 || head_dim <= 0)
    return NPO_BAD_ARG;
  for (int32_t r = 0; r < rows; ++r) {
    for (int32_t h = 0; h < q_heads; ++h) {
      int64_t rh = (int64_t)r * q_heads + h;
      const double* lse = lse_part + rh * num_splits;
      double* o = out + rh * head_dim;
      double big = -INFINITY;
      for (int32_t s = 0; s < num_splits; ++s)
        if (lse[s] > big) big = lse[s];
      for (int32_t d = 0; d < head_dim; ++d) o[d] = 0.0;
      if (big == -INFINITY) continue;
      double wsum = 0.0;
      for (int32_t s = 0; s < num_splits; ++s) {
        if (lse[s] == -INFINITY) continue;
        double w = exp(lse[s] - big);
        wsum += w;
        const double* os = o_part + (rh * num_splits + s) * head_dim;
        for (int32_t d = 0; d < head_dim; ++d) o[d] += w * os[d];
      }
      for (int32_t d = 0; d < head_dim; ++d) o[d] /= wsum;
    }
  }
  return NPO_OK;
}
