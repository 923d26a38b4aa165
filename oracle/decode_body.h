/*
 * decode_body.h -- the oracle's decode read, written once and included by
 * np_oracle.c for each working precision (NPO_REAL = double or float).
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE (see np_oracle.c).
 *
 * For each row r, kv head kh, query token i < query_len, query head h of
 * that kv head's group and split s:
 *   1. gather: for t < context_lens[r], K_t and V_t are the [head_dim]
 *      vectors at pool slot block_tables[r][t / bs] * bs + t % bs, kv head
 *      kh ("Day 17: paging under the sampling path", Diagram: a block table
 *      maps tokens to blocks; "Day 25: the fused read dispatches to the
 *      kernel backend", What I added today: attention over the gathered slots);
 *   2. scores: s_t = scale * sum_d q[r, i, h, d] * K_t[d], over the split's
 *      tokens t in [s * split_len, min((s + 1) * split_len, e)), where
 *      e = c - query_len + i + 1: query token i is the row's position
 *      c - query_len + i and the causal softmax lets it see history
 *      positions up to its own ("Day 25", What I learned 1: the reference
 *      softmax is causal, in fp32, position by position).  With query_len = 1, e = c: the whole
 *      history.  Several query tokens per row are the query_len axis of the
 *      read's score shape rows * heads * query_len * width ("Day 60: the
 *      read becomes a choice", What I learned 5);
 *   3. exact two-pass softmax by index: m = max_t s_t,
 *      p_t = exp(s_t - m), Z = sum_t p_t ("Day 25", What I learned 1);
 *   4. out = sum_t p_t V_t / Z and lse = m + log Z.
 * An empty split (no tokens) gives out = 0 and lse = -inf.  With
 * num_splits = 1 and split_len >= the context this is the whole read.
 *
 * Layouts (all dense, row-major):
 *   q            [rows, query_len, q_heads, head_dim] storage dtype
 *   k/v_pool     [num_blocks, block_size, kv_heads, head_dim]
 *   block_tables [rows, max_blocks_per_row] int32 (entries past the row's
 *                last needed block are never read)
 *   context_lens [rows] int32
 *   out          [rows, query_len, q_heads, num_splits, head_dim]  NPO_REAL
 *   lse          [rows, query_len, q_heads, num_splits]            NPO_REAL
 */

int NPO_NAME(npo_paged_decode)(
    NPO_REAL* out, NPO_REAL* lse, const void* q, const void* k_pool,
    const void* v_pool, int dtype, int64_t num_blocks, int32_t block_size,
    int32_t kv_heads, int32_t head_dim, const int32_t* block_tables,
    int32_t max_blocks_per_row, const int32_t* context_lens, int32_t rows,
    int32_t query_len, int32_t q_heads, double scale, int64_t split_len,
    int32_t num_splits) {
  if (npo_elem_size(dtype) == 0 || num_blocks <= 0 || block_size <= 0 ||
      kv_heads <= 0 || head_dim <= 0 || max_blocks_per_row < 0 || rows < 0 ||
      query_len <= 0 || q_heads <= 0 || q_heads % kv_heads != 0 ||
      split_len <= 0 || num_splits <= 0)
    return NPO_BAD_ARG;
  const int32_t group = q_heads / kv_heads;
  const NPO_REAL sc = (NPO_REAL)scale;
  const int64_t capacity = (int64_t)max_blocks_per_row * block_size;

  for (int32_t r = 0; r < rows; ++r) {
    const int64_t c = context_lens[r];
    if (c < 0 || c > capacity) return NPO_BAD_CONTEXT;
    if (c > split_len * (int64_t)num_splits) return NPO_BAD_ARG;

    for (int32_t kh = 0; kh < kv_heads; ++kh) {
      /* 1. gather this row's history for kv head kh into contiguous arrays */
      size_t n = (size_t)(c > 0 ? c : 1);
      NPO_REAL* hk = (NPO_REAL*)malloc(n * (size_t)head_dim * sizeof(NPO_REAL));
      NPO_REAL* hv = (NPO_REAL*)malloc(n * (size_t)head_dim * sizeof(NPO_REAL));
      NPO_REAL* sco = (NPO_REAL*)malloc(n * sizeof(NPO_REAL));
      if (!hk || !hv || !sco) {
        free(hk);
        free(hv);
        free(sco);
        return NPO_NO_MEMORY;
      }
      for (int64_t t = 0; t < c; ++t) {
        int64_t block = block_tables[(int64_t)r * max_blocks_per_row + t / block_size];
        if (block < 0 || block >= num_blocks) {
          free(hk);
          free(hv);
          free(sco);
          return NPO_BAD_BLOCK;
        }
        int64_t slot = block * block_size + t % block_size;
        for (int32_t d = 0; d < head_dim; ++d) {
          int64_t idx = (slot * kv_heads + kh) * head_dim + d;
          hk[t * head_dim + d] = (NPO_REAL)npo_load(k_pool, dtype, idx);
          hv[t * head_dim + d] = (NPO_REAL)npo_load(v_pool, dtype, idx);
        }
      }

      for (int32_t qi = 0; qi < query_len; ++qi)
      for (int32_t h = kh * group; h < (kh + 1) * group; ++h) {
        /* query token qi sees history positions [0, e) */
        int64_t e = c - query_len + qi + 1;
        if (e < 0) e = 0;
        int64_t rq = (int64_t)r * query_len + qi;
        for (int32_t s = 0; s < num_splits; ++s) {
          int64_t rhs = (rq * q_heads + h) * num_splits + s;
          NPO_REAL* o = out + rhs * head_dim;
          int64_t tb = (int64_t)s * split_len;
          int64_t te = tb + split_len < e ? tb + split_len : e;
          for (int32_t d = 0; d < head_dim; ++d) o[d] = 0;
          if (tb >= te) {
            lse[rhs] = -INFINITY;
            continue;
          }
          /* 2. scores */
          for (int64_t t = tb; t < te; ++t) {
            NPO_REAL dot = 0;
            for (int32_t d = 0; d < head_dim; ++d) {
              NPO_REAL qd = (NPO_REAL)npo_load(
                  q, dtype, (rq * q_heads + h) * head_dim + d);
              dot += qd * hk[t * head_dim + d];
            }
            sco[t] = sc * dot;
          }
          /* 3. exact softmax: max, exponentials, their sum */
          NPO_REAL m = sco[tb];
          for (int64_t t = tb + 1; t < te; ++t)
            if (sco[t] > m) m = sco[t];
          NPO_REAL z = 0;
          for (int64_t t = tb; t < te; ++t) {
            sco[t] = NPO_EXP(sco[t] - m);
            z += sco[t];
          }
          /* 4. probability-weighted sum of V, and the log-sum-exp */
          for (int64_t t = tb; t < te; ++t)
            for (int32_t d = 0; d < head_dim; ++d)
              o[d] += sco[t] * hv[t * head_dim + d];
          for (int32_t d = 0; d < head_dim; ++d) o[d] /= z;
          lse[rhs] = m + NPO_LOG(z);
        }
      }
      free(hk);
      free(hv);
      free(sco);
    }
  }
  return NPO_OK;
}
