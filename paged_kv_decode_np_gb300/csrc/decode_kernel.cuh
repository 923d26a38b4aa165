// decode_kernel.cuh -- what every decode kernel of the library shares: the
// launch parameters, the fused append, the stage geometry of the bf16 read.
//
// The operation (per row r, query head h, kv head h / G): attention of the
// row's query token over its whole history, the history gathered through the
// row's block table from a pool [num_blocks, block_size, kv_heads, head_dim]
// ("Day 17: paging under the sampling path", Diagram; "Day 25: the fused
// read dispatches to the kernel backend", What I added today).  The softmax
// is streamed: a running max m and sum l per head, the accumulator rescaled
// by 2^(m_old - m_new) whenever the max grows, so no full array of scores is
// ever built ("Day 60: the read becomes a choice", What I added today and
// Post angle; "Day 25", Why it matters: the streamed softmax sums the
// exponentials in another order, so results are close to, not bit-equal
// with, the exact softmax).  Scores are kept in log2 units (q, or the QK
// product, scaled by scale*log2(e)) so the exponentials are single ex2
// instructions.
//
// The kernels (GB300 design, not from the pages): a producer warp walks the
// block table and moves K/V with TMA into an mbarrier ring of shared-memory
// stages; consumer warps, one per kv head (or several per head taking
// alternate stages), compute for all G query heads of the head's group, so
// one K/V fetch serves the whole group.
//   * decode_mma.cuh: bf16 pools on the tensor cores, split grid
//     (num_splits, rows, kv_heads / HG).
//   * decode_fma.cuh: fp32 pools on the FMA pipes, split grid.
//   * decode_stream.cuh: the balanced read (one CTA per SM over all rows,
//     either consumer) and its merge of the rows cut between CTAs.
#pragma once

#include <math.h>

#include "np_common.cuh"

namespace npk {

struct DecodeParams {
  // Tiled TMA maps of the K and V pools as [head_dim, slot, kv_head] with the
  // kv-head stride innermost after head_dim's (see decode_mma.cuh); only
  // read when use_tmap is set.
  CUtensorMap tm_k;
  CUtensorMap tm_v;
  void* out;             // [R, Hq, D] T, when num_splits == 1
  float* ws_o;           // [R, Hq, S, D] fp32, when num_splits > 1
  float* ws_lse;         // [R, Hq, S] fp32 (natural log)
  const void* q;         // [R, Hq, D] T
  const void* k_pool;    // [NB, bs, Hk, D] T
  const void* v_pool;
  const int32_t* block_tables;  // [R, MB]
  const int32_t* context_lens;  // [R]
  int32_t* err;
  int64_t num_blocks;
  int64_t split_len;     // tokens per split
  int32_t block_size;
  int32_t kv_heads;
  int32_t head_group;    // HG: kv heads per CTA (divides kv_heads)
  int32_t token_warps;   // TW: consumer warps per kv head
  int32_t stage_slices;  // balanced read: K::CT-token pieces per warp and stage (SL)
  int32_t max_blocks_per_row;
  int32_t q_heads;
  int32_t num_splits;
  int32_t stages;        // ring depth
  int32_t use_tmap;      // 1: K/V arrive through tm_k/tm_v boxes
  int32_t box_tokens;    // tokens per TMA box (divides block_size and the chunk)
  int32_t query_len;     // query tokens per row (the last query_len positions)
  float qscale;          // softmax scale * log2(e)
  // Fused append (np_paged_append_decode): row r's new K/V rows, token j to
  // pool slot slot_mapping[r*Q + j], written by the CTA whose split holds
  // position context_lens[r] - Q + j, before that CTA reads it.  Null when
  // not fused.
  const void* k_new;     // [R, Q, Hk, D] T
  const void* v_new;
  const int64_t* slot_mapping;  // [R, Q]
  // Balanced streamed read (num_splits == 0; decode_stream.cuh): partials
  // go to ws_o, each CTA's merge descriptor to st_desc ([P][4]).
  int32_t rows;
  int32_t* st_desc;
};

// Fused append, run by every thread of the CTA before its pipeline starts.
// Row r's Q new tokens are its positions c - Q .. c - 1.  The CTA whose token
// range [t0, t1) holds new token j's position writes its HG heads' slice of
// that token's K and V rows to the slot the row's block table gives the
// position -- the slot mapping must name that same slot (a negative entry
// means "no new token"); an entry that does not is flagged (NP_FLAG_SLOT)
// and nothing is written, so no other CTA can read a slot being written.
// The generic-proxy stores are made visible to this CTA's TMA (async-proxy)
// reads by fence.proxy.async before the barrier that precedes the first copy.
template <int D, int ES>
__device__ __forceinline__ void fused_append(const DecodeParams& p, int r, int hgi, int HG,
                                             int64_t c, int64_t t0, int64_t t1,
                                             int tid = threadIdx.x, int nthreads = blockDim.x) {
  if (p.slot_mapping == nullptr) return;
  const int Q = p.query_len;
  bool wrote = false;
  for (int j = 0; j < Q; ++j) {
    const int64_t pos = c - Q + j;
    if (pos < 0 || pos < t0 || pos >= t1) continue;
    const int64_t rq = (int64_t)r * Q + j;
    const int64_t nvec = (int64_t)HG * D * ES / 16;  // 16-byte vectors of the slice
    const int64_t src0 = (rq * p.kv_heads + (int64_t)hgi * HG) * D * ES / 16;
    const uint4* kn = static_cast<const uint4*>(p.k_new);
    const uint4* vn = static_cast<const uint4*>(p.v_new);
    // the slot, its table entry and this thread's first vectors are loaded
    // together (one round trip, not three in a chain): at the kernel's start
    // the read's own copies load the memory system
    const bool first = tid < nvec;
    uint4 k0 = make_uint4(0, 0, 0, 0), v0 = k0;
    if (first) {
      k0 = kn[src0 + tid];
      v0 = vn[src0 + tid];
    }
    const int64_t bs = p.block_size;
    const int64_t s = p.slot_mapping[rq];
    const int64_t b = p.block_tables[(int64_t)r * p.max_blocks_per_row + pos / bs];
    if (s < 0) continue;
    if (b < 0 || b >= p.num_blocks || s != b * bs + pos % bs) {
      if (tid == 0) set_flag(p.err, NP_FLAG_SLOT);
      continue;
    }
    const int64_t dst0 = (s * p.kv_heads + (int64_t)hgi * HG) * D * ES / 16;
    uint4* kd = static_cast<uint4*>(const_cast<void*>(p.k_pool));
    uint4* vd = static_cast<uint4*>(const_cast<void*>(p.v_pool));
    if (first) {
      kd[dst0 + tid] = k0;
      vd[dst0 + tid] = v0;
    }
    for (int64_t i = tid + nthreads; i < nvec; i += nthreads) {
      kd[dst0 + i] = kn[src0 + i];
      vd[dst0 + i] = vn[src0 + i];
    }
    wrote = true;
  }
  if (wrote) asm volatile("fence.proxy.async.global;" ::: "memory");
}

// One new token of the fused append, written by a group of `tpt` threads
// (thread t of the group): row r's token j (position pos), the HG heads of
// group hgi.  Same rule as fused_append.  The slot, its table entry and the
// thread's vectors of K and of V (at most kAppendVpl of each: the caller
// sizes the group so) are loaded together -- one round trip -- so the
// groups of a CTA append their tokens side by side in about the time of
// one.  Returns whether the thread stored anything (the caller fences
// before the barrier that precedes its TMA reads).
constexpr int kAppendVpl = 4;
template <int D, int ES>
__device__ __forceinline__ bool append_token_group(const DecodeParams& p, int r, int hgi, int HG,
                                                   int64_t pos, int j, int t, int tpt) {
  const int64_t rq = (int64_t)r * p.query_len + j;
  const int nvec = HG * D * ES / 16;  // 16-byte vectors of the slice
  const int64_t src0 = (rq * p.kv_heads + (int64_t)hgi * HG) * D * ES / 16;
  const uint4* kn = static_cast<const uint4*>(p.k_new);
  const uint4* vn = static_cast<const uint4*>(p.v_new);
  uint4 kr[kAppendVpl], vr[kAppendVpl];
#pragma unroll
  for (int e = 0; e < kAppendVpl; ++e) {
    const int i = t + tpt * e;
    if (i < nvec) {
      kr[e] = kn[src0 + i];
      vr[e] = vn[src0 + i];
    }
  }
  const int64_t bs = p.block_size;
  const int64_t s = p.slot_mapping[rq];
  const int64_t b = p.block_tables[(int64_t)r * p.max_blocks_per_row + pos / bs];
  if (s < 0) return false;
  if (b < 0 || b >= p.num_blocks || s != b * bs + pos % bs) {
    if (t == 0) set_flag(p.err, NP_FLAG_SLOT);
    return false;
  }
  const int64_t dst0 = (s * p.kv_heads + (int64_t)hgi * HG) * D * ES / 16;
  uint4* kd = static_cast<uint4*>(const_cast<void*>(p.k_pool));
  uint4* vd = static_cast<uint4*>(const_cast<void*>(p.v_pool));
#pragma unroll
  for (int e = 0; e < kAppendVpl; ++e) {
    const int i = t + tpt * e;
    if (i < nvec) {
      kd[dst0 + i] = kr[e];
      vd[dst0 + i] = vr[e];
    }
  }
  return t < nvec;
}

#ifndef NPK_MMA_CT
#define NPK_MMA_CT 16  // tokens per pipeline stage for 64 <= head_dim < 256
#endif

// Tokens per pipeline stage of the bf16 tensor-core read (host and device
// agree on it: a TMA box never holds more tokens than a stage).  A stage
// holds about 64 KB of K+V at 8 kv heads.
__host__ __device__ constexpr int mma_chunk_tokens(int head_dim) {
  return head_dim >= 256 ? 8 : (head_dim >= 64 ? NPK_MMA_CT : 32);
}

constexpr int kMaxConsumerWarps = 8;
constexpr int kMaxThreads = 32 * (kMaxConsumerWarps + 1);

}  // namespace npk
