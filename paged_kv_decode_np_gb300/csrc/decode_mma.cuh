// decode_mma.cuh -- the paged decode read for bf16 pools on the tensor cores
// (warp-level mma.sync m16n8k16, bf16 inputs, fp32 accumulation).
//
// Same operation, grid and pipeline roles as decode_kernel.cuh (see there for
// the citations): a producer warp walks the block table and moves K/V with
// TMA into an mbarrier ring; consumer warp (hl, tw) owns kv head hl and the G
// query heads of its group.  The consumer's arithmetic is a pair of small
// dense products per 16-token tile:
//
//   S^T[h, t] = q[h, :] . K[t, :]      M = 16 query heads (G real, rest 0),
//                                      N = 8 tokens, K = 16 dims per mma;
//                                      q fragments live in registers, K^T
//                                      fragments come from ldmatrix.
//   O^T[d, h] += V[t, d]^T P[h, t]^T   M = 16 dims, N = 8 heads, K = 16
//                                      tokens; V^T fragments from
//                                      ldmatrix.trans, and P^T is the S^T
//                                      accumulator itself, rounded to bf16
//                                      (the C layout of S^T is the B layout
//                                      of P^T), so P never touches memory.
//
// With several query tokens per row (query_len Q, G*Q <= 16) the mma rows
// are (query token, head) pairs, row = qi*G + h: one K/V fetch serves every
// query token of the group; rows 8..15 use the second PV n-tile (TWO).  A
// query token at position c - Q + qi only sees positions up to its own.
//
// Scores leave the tensor cores in fp32 and are scaled by scale*log2(e) there
// (q stays exactly the stored bf16).  The online softmax keeps a running max
// and sum per head in fp32; the 4 lanes that hold one head's scores reduce
// with two xor-shuffles.  P is rounded to bf16 for the PV product (relative
// error 2^-9 per weight; the accumulation stays fp32).
//
// Staging (how a chunk of CT tokens x HG kv heads lands in shared memory):
//  * TMAP (head_dim a multiple of 64): tiled TMA boxes of {64 dims, B tokens,
//    HG heads} from a tensor map whose dimensions are (dim, slot, kv head) --
//    so inside a box each head's B token rows are consecutive 128-byte rows,
//    stored with the 128-byte swizzle.  The 8 token rows one ldmatrix phase
//    reads then sit in 8 different bank groups.  A 64 KB chunk is 4 copies.
//  * otherwise: one 1-D bulk copy per token row, to a row stride padded by
//    16 bytes (the same conflict-free property, more copy instructions).
#pragma once

#include <math.h>

#include "decode_kernel.cuh"

namespace npk {

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                          uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// D = A*B + D, m16n8k16, bf16 x bf16 -> fp32
__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

#ifndef NPK_MMA_MIN_BLOCKS
#define NPK_MMA_MIN_BLOCKS 1  // resident CTAs per SM the register budget targets
#endif

constexpr int kMmaRows = 16;  // mma M: (query token, head) rows per kv head

template <int D, int G, bool TMAP>
struct MmaCfg {
  static constexpr int KS = D / 16;  // mma k-steps over head_dim (QK), m-tiles (PV)
  static constexpr int ST = 16;      // tokens per softmax tile
  static constexpr int CT = mma_chunk_tokens(D);  // tokens per stage
  // CT < ST is allowed: the tile's rows past the chunk are masked and their
  // shared-memory reads are redirected to the tile's first row.
  static_assert(D % 16 == 0 && G >= 0 && G <= 16, "shape");  // G = 0: set at run time
  static_assert((CT % ST == 0 || ST % CT == 0) && CT <= 32, "tiling");
  static_assert(!TMAP || D % 64 == 0, "TMA boxes are 64 dims wide");
};

template <int D, int G, bool TMAP>
struct MmaSmem {
  using C = MmaCfg<D, G, TMAP>;
  // bytes between consecutive token rows (padded layout only)
  __host__ __device__ static constexpr size_t row_stride(int hg) { return (size_t)hg * D * 2 + 16; }
  __host__ __device__ static constexpr size_t stage_bytes(int hg) {
    return TMAP ? 2ull * C::CT * hg * D * 2 : 2ull * C::CT * row_stride(hg);
  }
  __host__ __device__ static constexpr size_t merge_bytes(int warps) {
    return (size_t)warps * kMmaRows * (D + 2) * sizeof(float);
  }
  __host__ __device__ static constexpr size_t ring_bytes(int hg, int stages, int warps) {
    size_t ring = stage_bytes(hg) * stages;
    size_t m = merge_bytes(warps);
    return ((ring > m ? ring : m) + 1023) / 1024 * 1024;
  }
  // + 1024: the ring starts at the first 1024-byte boundary of the window
  __host__ __device__ static constexpr size_t total(int hg, int stages, int warps) {
    return 1024 + ring_bytes(hg, stages, warps) + 16ull * stages + 16;
  }
};

// One online-softmax row update for a 4-score slice (two token pairs) held by
// the 4 lanes of a fragment row group.  Returns alpha (the rescale of the
// row's running output); writes the probabilities into sc.  A row with no
// visible token yet keeps m = -inf and gets alpha = p = 0 (no -inf - -inf).
__device__ __forceinline__ float softmax_row(float (&sc)[4], float& m_run, float& l_run) {
  constexpr unsigned FULL = 0xffffffffu;
  float mt = fmaxf(fmaxf(sc[0], sc[1]), fmaxf(sc[2], sc[3]));
  mt = fmaxf(mt, __shfl_xor_sync(FULL, mt, 1));
  mt = fmaxf(mt, __shfl_xor_sync(FULL, mt, 2));
  const float mn = fmaxf(m_run, mt);
  const float mref = (mn == -INFINITY) ? 0.f : mn;
  const float alpha = ex2(m_run - mref);
  m_run = mn;
#pragma unroll
  for (int e = 0; e < 4; ++e) sc[e] = ex2(sc[e] - mref);
  l_run = fmaf(l_run, alpha, (sc[0] + sc[1]) + (sc[2] + sc[3]));
  return alpha;
}

// Where one kv head's rows of a stage live in shared memory, and the address
// of the 16-byte chunk of dims [16*ks + 8*ld_c, +8) of a token row.
template <int D, bool TMAP>
struct StageLayout {
  int BT;               // tokens per TMA box
  uint32_t slab_bytes;  // one 64-dim slab of a box: HG heads x BT rows of 128 bytes (TMAP)
  uint32_t box_bytes;   // one box: D/64 slabs (TMAP)
  uint32_t RS;          // token-row stride (per-token copies)
  int hl;               // kv head within the CTA's group

  __device__ __forceinline__ void row(int tok, uint32_t& off, uint32_t& swz) const {
    if constexpr (TMAP) {
      const int bx = tok / BT, tr = tok - bx * BT;
      off = bx * box_bytes + (hl * BT + tr) * 128;
      swz = (off >> 7) & 7;
    } else {
      off = tok * RS + hl * D * 2;
      swz = 0;
    }
  }
  __device__ __forceinline__ uint32_t chunk(uint32_t base, int ks, uint32_t off, uint32_t swz,
                                            int ld_c) const {
    if constexpr (TMAP) {
      const uint32_t cidx = ((2 * ks) & 7) + ld_c;  // chunk within the 128-byte row
      return base + (ks >> 2) * slab_bytes + off + ((cidx ^ swz) << 4);
    } else {
      return base + off + ks * 32 + ld_c * 16;
    }
  }
};

// Producer: issue the copies of one chunk -- tokens [cb, cb + n) of row r,
// kv heads [hgi*HG, (hgi+1)*HG) -- completing on `fb`.  The row's block ids
// are fetched 32 at a time into `my_id` (window starting at logical block
// `win`; win < 0 forces a fetch) and broadcast with shuffles.
template <int D, bool TMAP>
__device__ __forceinline__ void produce_chunk(const DecodeParams& p, const StageLayout<D, TMAP>& L,
                                              int64_t r, int hgi, int HG, int64_t cb, int n,
                                              int64_t nblk, uint32_t kdst, uint32_t vdst,
                                              uint32_t fb, uint64_t pol, int64_t& win,
                                              int32_t& my_id, int lane) {
  constexpr unsigned FULL = 0xffffffffu;
  const int64_t bs = p.block_size;
  const uint32_t row_bytes = (uint32_t)HG * D * 2;
  const int64_t jfirst = cb / bs;
  const int64_t jlast = (cb + n - 1) / bs;
  if (win < 0 || jfirst < win || jlast >= win + 32) {
    win = jfirst;
    const int64_t jj = win + lane;
    my_id = jj < nblk ? p.block_tables[r * p.max_blocks_per_row + jj] : 0;
  }
  if constexpr (TMAP) {
    // boxes of BT tokens x HG heads x all D/64 slabs; each lies inside one
    // block (BT divides the block size and the chunk start) and is copied
    // whole (rows past the history are masked by the consumers)
    const int nbox = (n + L.BT - 1) / L.BT;
    if (lane == 0) mbar_arrive_expect_tx(fb, 2u * nbox * L.box_bytes);
    const int items = nbox * 2;  // (box, K|V)
    const int rounds = (items + 31) / 32;
    for (int rd = 0; rd < rounds; ++rd) {
      const int it = rd * 32 + lane;
      const int bx = (it < items ? it : 0) >> 1;
      const int64_t t = cb + (int64_t)bx * L.BT;
      const int64_t j = t / bs;
      int64_t b = __shfl_sync(FULL, my_id, (int)(j - win));
      if (it < items) {
        const bool isv = (it & 1) != 0;
        if (b < 0 || b >= p.num_blocks) {
          set_flag(p.err, NP_FLAG_BLOCK_ID);
          b = 0;
        }
        const int64_t slot = b * bs + (t - j * bs);
        const uint32_t dst = (isv ? vdst : kdst) + bx * L.box_bytes;
        tma_load_4d(dst, isv ? &p.tm_v : &p.tm_k, 0, (int32_t)slot, hgi * HG, 0, fb, pol);
      }
    }
  } else {
    if (lane == 0) mbar_arrive_expect_tx(fb, 2u * (uint32_t)n * row_bytes);
    const int64_t t = cb + (lane < n ? lane : 0);
    const int64_t j = t / bs;
    int64_t b = __shfl_sync(FULL, my_id, (int)(j - win));
    if (b < 0 || b >= p.num_blocks) {
      if (lane < n) set_flag(p.err, NP_FLAG_BLOCK_ID);
      b = 0;
    }
    if (lane < n) {
      const int64_t slot = b * bs + (t - j * bs);
      const int64_t pool_row = (int64_t)p.kv_heads * D * 2;
      const char* kp = static_cast<const char*>(p.k_pool) + (int64_t)hgi * row_bytes;
      const char* vp = static_cast<const char*>(p.v_pool) + (int64_t)hgi * row_bytes;
      bulk_g2s(kdst + lane * L.RS, kp + slot * pool_row, row_bytes, fb, pol);
      bulk_g2s(vdst + lane * L.RS, vp + slot * pool_row, row_bytes, fb, pol);
    }
  }
}

// One consumer warp's read of one kv head: q fragments, the running softmax
// of its two fragment rows (g4 and g4 + 8) and the O^T accumulators.
template <int D, int G, bool TWO>
struct MmaWarp {
  static constexpr int KS = D / 16;
  uint32_t qa0[KS], qa2[KS], qa1[TWO ? KS : 1], qa3[TWO ? KS : 1];
  float mA, lA, mB, lB;
  // O^T fragments: rows d = 16*mi + lane/4 (+8); columns = mma rows
  // 2*(lane%4) (+1) in oA, 8 + 2*(lane%4) (+1) in oB
  float oA[KS][4];
  float oB[TWO ? KS : 1][4];
  // last position each row may see (-1: a padding row); positions fit int32
  // (context_lens are int32)
  int32_t limA, limB;
  int gr;              // query heads per kv head (G, or q_heads/kv_heads when G = 0)

  // q of row r, kv head kvh: mma row qi*G + h is query token qi, head
  // kvh*G + h; rows >= G*Q are zero.  Resets the softmax state.
  __device__ __forceinline__ void begin(const DecodeParams& p, int64_t r, int kvh, int64_t c,
                                        int lane) {
    gr = G > 0 ? G : p.q_heads / p.kv_heads;
    const int Q = p.query_len, MR = gr * Q;
    const int g4 = lane >> 2, c4 = lane & 3;
    auto qrow = [&](int row) -> const __nv_bfloat16* {
      const int qi = row / gr, h = row - (row / gr) * gr;
      return static_cast<const __nv_bfloat16*>(p.q) +
             ((r * Q + qi) * p.q_heads + kvh * gr + h) * D;
    };
    const bool liveA = g4 < MR, liveB = g4 + 8 < MR;
    limA = liveA ? (int32_t)(c - Q + g4 / gr) : -1;
    limB = liveB ? (int32_t)(c - Q + (g4 + 8) / gr) : -1;
    const __nv_bfloat16* qa = liveA ? qrow(g4) : nullptr;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      qa0[ks] = liveA ? *reinterpret_cast<const uint32_t*>(qa + 16 * ks + 2 * c4) : 0u;
      qa2[ks] = liveA ? *reinterpret_cast<const uint32_t*>(qa + 16 * ks + 8 + 2 * c4) : 0u;
    }
    if constexpr (TWO) {
      const __nv_bfloat16* qb = liveB ? qrow(g4 + 8) : nullptr;
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        qa1[ks] = liveB ? *reinterpret_cast<const uint32_t*>(qb + 16 * ks + 2 * c4) : 0u;
        qa3[ks] = liveB ? *reinterpret_cast<const uint32_t*>(qb + 16 * ks + 8 + 2 * c4) : 0u;
      }
    }
    mA = mB = -INFINITY;
    lA = lB = 0.f;
#pragma unroll
    for (int mi = 0; mi < KS; ++mi)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        oA[mi][e] = 0.f;
        if constexpr (TWO) oB[mi][e] = 0.f;
      }
  }

  // One tile: up to 16 tokens from tile-local token sb of a staged chunk
  // (K rows at kst, V rows at vst) whose first token is position tch and
  // whose first nvalid tokens are valid.
  template <bool TMAP>
  __device__ __forceinline__ void tile(const StageLayout<D, TMAP>& L, uint32_t kst, uint32_t vst,
                                       int sb, int nvalid, int64_t tch, float qscale, int lane) {
    constexpr unsigned FULL = 0xffffffffu;
    const int c4 = lane & 3;
    // ldmatrix lane addressing: matrix (lane/8) covers tokens 8*(lane/16) +
    // (0..7) and the 8-dim column chunk (lane/8)%2 of a 16-dim step; the same
    // pattern serves K (B of QK) and V (A of PV, transposed load).  Rows past
    // the valid tokens read row sb instead (finite data; probability 0).
    const int ld_tok = ((lane >> 4) << 3) + (lane & 7);
    const int ld_c = (lane >> 3) & 1;
    const int tok = (sb + ld_tok < nvalid) ? sb + ld_tok : sb;
    uint32_t off, swz;
    L.row(tok, off, swz);
    // ---- S^T = q K^T for 16 tokens (two n-tiles of 8)
    float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      uint32_t b0, b1, b2, b3;
      ldsm_x4(L.chunk(kst, ks, off, swz, ld_c), b0, b1, b2, b3);
      if constexpr (TWO) {
        mma_bf16(s0, qa0[ks], qa1[ks], qa2[ks], qa3[ks], b0, b1);
        mma_bf16(s1, qa0[ks], qa1[ks], qa2[ks], qa3[ks], b2, b3);
      } else {
        mma_bf16(s0, qa0[ks], 0u, qa2[ks], 0u, b0, b1);
        mma_bf16(s1, qa0[ks], 0u, qa2[ks], 0u, b2, b3);
      }
    }
    // ---- masks: token (tile-local) 2*c4 + {0, 1, 8, 9} must be a valid
    // token of the chunk and at or before the row's own position
    // (limits relative to the chunk's first position: no overflow, as
    // 0 <= tch <= INT32_MAX and lim >= -1)
    const int lt = sb + 2 * c4;
    const int32_t relA = limA - (int32_t)tch;
    const bool v0 = lt < nvalid, v1 = lt + 1 < nvalid, v8 = lt + 8 < nvalid, v9 = lt + 9 < nvalid;
    float sa[4] = {s0[0] * qscale, s0[1] * qscale, s1[0] * qscale, s1[1] * qscale};
    if (!(v0 && lt <= relA)) sa[0] = -INFINITY;
    if (!(v1 && lt + 1 <= relA)) sa[1] = -INFINITY;
    if (!(v8 && lt + 8 <= relA)) sa[2] = -INFINITY;
    if (!(v9 && lt + 9 <= relA)) sa[3] = -INFINITY;
    const float alphaA = softmax_row(sa, mA, lA);
    const uint32_t pa0 = pack_bf16(sa[0], sa[1]);
    const uint32_t pa1 = pack_bf16(sa[2], sa[3]);
    float alphaB = 1.f;
    uint32_t pb0 = 0u, pb1 = 0u;
    if constexpr (TWO) {
      float sbv[4] = {s0[2] * qscale, s0[3] * qscale, s1[2] * qscale, s1[3] * qscale};
      const int32_t relB = limB - (int32_t)tch;
      if (!(v0 && lt <= relB)) sbv[0] = -INFINITY;
      if (!(v1 && lt + 1 <= relB)) sbv[1] = -INFINITY;
      if (!(v8 && lt + 8 <= relB)) sbv[2] = -INFINITY;
      if (!(v9 && lt + 9 <= relB)) sbv[3] = -INFINITY;
      alphaB = softmax_row(sbv, mB, lB);
      pb0 = pack_bf16(sbv[0], sbv[1]);
      pb1 = pack_bf16(sbv[2], sbv[3]);
    }
    // ---- rescale O^T columns (mma rows 2*c4, 2*c4+1 and +8) when a max moved
    if (__any_sync(FULL, alphaA != 1.f || alphaB != 1.f)) {
      const float a_lo = __shfl_sync(FULL, alphaA, 8 * c4);
      const float a_hi = __shfl_sync(FULL, alphaA, 8 * c4 + 4);
#pragma unroll
      for (int mi = 0; mi < KS; ++mi) {
        oA[mi][0] *= a_lo;
        oA[mi][1] *= a_hi;
        oA[mi][2] *= a_lo;
        oA[mi][3] *= a_hi;
      }
      if constexpr (TWO) {
        const float b_lo = __shfl_sync(FULL, alphaB, 8 * c4);
        const float b_hi = __shfl_sync(FULL, alphaB, 8 * c4 + 4);
#pragma unroll
        for (int mi = 0; mi < KS; ++mi) {
          oB[mi][0] *= b_lo;
          oB[mi][1] *= b_hi;
          oB[mi][2] *= b_lo;
          oB[mi][3] *= b_hi;
        }
      }
    }
    // ---- O^T += V^T P^T
#pragma unroll
    for (int mi = 0; mi < KS; ++mi) {
      uint32_t a0, a1, a2, a3;
      ldsm_x4_t(L.chunk(vst, mi, off, swz, ld_c), a0, a1, a2, a3);
      mma_bf16(oA[mi], a0, a1, a2, a3, pa0, pa1);
      if constexpr (TWO) mma_bf16(oB[mi], a0, a1, a2, a3, pb0, pb1);
    }
  }

  // each row's sum over its 4 lanes
  __device__ __forceinline__ void finish() {
    constexpr unsigned FULL = 0xffffffffu;
    lA += __shfl_xor_sync(FULL, lA, 1);
    lA += __shfl_xor_sync(FULL, lA, 2);
    lB += __shfl_xor_sync(FULL, lB, 1);
    lB += __shfl_xor_sync(FULL, lB, 2);
  }

  // The whole row's normalised output: mma row qi*G + h to out[r, qi,
  // kvh*G + h] (bf16), rows >= G*Q skipped.  After finish().  Each lane
  // writes four rows at most (2*c4, 2*c4 + 1 and, with TWO, 8 more): their
  // addresses and reciprocal sums are formed once.
  __device__ __forceinline__ void store_out(const DecodeParams& p, int64_t r, int kvh,
                                            int lane) const {
    constexpr unsigned FULL = 0xffffffffu;
    const int Q = p.query_len, MR = gr * Q;
    const int g4 = lane >> 2, c4 = lane & 3;
    const float l_lo = __shfl_sync(FULL, lA, 8 * c4), l_hi = __shfl_sync(FULL, lA, 8 * c4 + 4);
    const float lb_lo = __shfl_sync(FULL, lB, 8 * c4), lb_hi = __shfl_sync(FULL, lB, 8 * c4 + 4);
    auto row_ptr = [&](int row) -> __nv_bfloat16* {
      if (row >= MR) return nullptr;
      const int qi = row / gr, h = row - qi * gr;
      return static_cast<__nv_bfloat16*>(p.out) +
             ((r * Q + qi) * p.q_heads + (int64_t)kvh * gr + h) * D;
    };
    auto inv = [](float l) { return l > 0.f ? 1.f / l : 0.f; };
    __nv_bfloat16* o0 = row_ptr(2 * c4);
    __nv_bfloat16* o1 = row_ptr(2 * c4 + 1);
    const float i0 = inv(l_lo), i1 = inv(l_hi);
#pragma unroll
    for (int mi = 0; mi < KS; ++mi) {
      const int d = 16 * mi + g4;
      if (o0) {
        o0[d] = __float2bfloat16_rn(oA[mi][0] * i0);
        o0[d + 8] = __float2bfloat16_rn(oA[mi][2] * i0);
      }
      if (o1) {
        o1[d] = __float2bfloat16_rn(oA[mi][1] * i1);
        o1[d + 8] = __float2bfloat16_rn(oA[mi][3] * i1);
      }
    }
    if constexpr (TWO) {
      __nv_bfloat16* o8 = row_ptr(8 + 2 * c4);
      __nv_bfloat16* o9 = row_ptr(9 + 2 * c4);
      const float i8 = inv(lb_lo), i9 = inv(lb_hi);
#pragma unroll
      for (int mi = 0; mi < KS; ++mi) {
        const int d = 16 * mi + g4;
        if (o8) {
          o8[d] = __float2bfloat16_rn(oB[mi][0] * i8);
          o8[d + 8] = __float2bfloat16_rn(oB[mi][2] * i8);
        }
        if (o9) {
          o9[d] = __float2bfloat16_rn(oB[mi][1] * i9);
          o9[d + 8] = __float2bfloat16_rn(oB[mi][3] * i9);
        }
      }
    }
  }

  // Unnormalised result rows into a [16 rows][D] fp32 array plus m and l
  // ([16] each) through the store st; rows >= MR are skipped.
  template <typename St = PlainStore>
  __device__ __forceinline__ void store_rows(float* m_out, float* l_out, float* o_out, int MR,
                                             int lane, St st = St()) const {
    const int g4 = lane >> 2;
    if ((lane & 3) == 0) {
      if (g4 < MR) {
        st(&m_out[g4], mA);
        st(&l_out[g4], lA);
      }
      if (TWO && g4 + 8 < MR) {
        st(&m_out[g4 + 8], mB);
        st(&l_out[g4 + 8], lB);
      }
    }
    const int c0 = 2 * (lane & 3);  // mma rows of this lane's O^T columns
#pragma unroll
    for (int mi = 0; mi < KS; ++mi) {
      const int d = 16 * mi + g4;
      if (c0 < MR) {
        st(&o_out[c0 * D + d], oA[mi][0]);
        st(&o_out[c0 * D + d + 8], oA[mi][2]);
      }
      if (c0 + 1 < MR) {
        st(&o_out[(c0 + 1) * D + d], oA[mi][1]);
        st(&o_out[(c0 + 1) * D + d + 8], oA[mi][3]);
      }
      if constexpr (TWO) {
        if (c0 + 8 < MR) {
          st(&o_out[(c0 + 8) * D + d], oB[mi][0]);
          st(&o_out[(c0 + 8) * D + d + 8], oB[mi][2]);
        }
        if (c0 + 9 < MR) {
          st(&o_out[(c0 + 9) * D + d], oB[mi][1]);
          st(&o_out[(c0 + 9) * D + d + 8], oB[mi][3]);
        }
      }
    }
  }
};

// The split grid's last step, for the consumer warp of kv head hl with
// tw = 0: the TW warps of that head left their unnormalised rows (m in log2
// units, l, O) in `merge` ([warp][m[16] l[16] O[16][D]] fp32); merge them
// (max and weights) and write each of the G*Q rows -- normalised to `out`
// (type T) for an unsplit read, else as this split's partial o and natural
// log lse.
template <typename T, int D>
__device__ __forceinline__ void split_write_rows(const DecodeParams& p, const float* merge,
                                                 int64_t r, int split, int kvh, int hl, int HG,
                                                 int TW, int Gr, int lane) {
  constexpr int RW = kMmaRows;
  const int stride_w = RW * (D + 2);
  const int Q = p.query_len, MR = Gr * Q;
  constexpr int DL = D >= 32 ? D / 32 : 1;  // dims per lane
  const int d0 = lane * DL;
  for (int row = 0; row < MR; ++row) {
    float mm = -INFINITY;
    for (int w2 = 0; w2 < TW; ++w2) mm = fmaxf(mm, merge[(hl + w2 * HG) * stride_w + row]);
    float ll = 0.f;
    float acc[DL];
#pragma unroll
    for (int e = 0; e < DL; ++e) acc[e] = 0.f;
    for (int w2 = 0; w2 < TW; ++w2) {
      const float* mg = merge + (hl + w2 * HG) * stride_w;
      const float a = (mg[row] == -INFINITY) ? 0.f : ex2(mg[row] - mm);
      ll = fmaf(mg[RW + row], a, ll);
      if (d0 < D) {
#pragma unroll
        for (int e = 0; e < DL; ++e) acc[e] = fmaf(mg[2 * RW + row * D + d0 + e], a, acc[e]);
      }
    }
    const int qi = row / Gr, h = row - qi * Gr;
    const int64_t rq = r * Q + qi;
    const int hq = kvh * Gr + h;
    const float inv = ll > 0.f ? 1.f / ll : 0.f;
    float ov[DL];
#pragma unroll
    for (int e = 0; e < DL; ++e) ov[e] = acc[e] * inv;
    if (d0 < D) {
      if (p.num_splits == 1) {
        T* orow = static_cast<T*>(p.out) + (rq * p.q_heads + hq) * D;
        Storage<T>::template store<DL>(orow + d0, ov);
      } else {
        const int64_t rs = (rq * p.q_heads + hq) * p.num_splits + split;
        float* orow = p.ws_o + rs * D + d0;
        if constexpr (DL >= 4) {
#pragma unroll
          for (int e = 0; e < DL; e += 4) Storage<float>::template store<4>(orow + e, ov + e);
        } else {
#pragma unroll
          for (int e = 0; e < DL; ++e) orow[e] = ov[e];
        }
        if (lane == 0)
          p.ws_lse[rs] = ll > 0.f ? mm * 0.69314718055994531f + logf(ll) : -INFINITY;
      }
    }
  }
}

template <int D, int G, bool TMAP, bool TWO>
__global__ void __launch_bounds__(kMaxThreads, NPK_MMA_MIN_BLOCKS)
    paged_decode_mma_kernel(const __grid_constant__ DecodeParams p) {
  using C = MmaCfg<D, G, TMAP>;
  using S = MmaSmem<D, G, TMAP>;
  constexpr unsigned FULL = 0xffffffffu;

  const int split = blockIdx.x;
  const int r = blockIdx.y;
  const int hgi = blockIdx.z;
  const int HG = p.head_group;
  const int TW = p.token_warps;
  const int NC = HG * TW;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int Gr = G > 0 ? G : p.q_heads / p.kv_heads;  // query heads per kv head
  const int hq0 = hgi * HG * Gr;
  const int Q = p.query_len;
  const int MR = Gr * Q;  // real mma rows (<= 16)

  const int64_t cap = (int64_t)p.max_blocks_per_row * p.block_size;
  int64_t c = p.context_lens[r];
  if (c < 0 || c > cap) {
    if (threadIdx.x == 0) set_flag(p.err, NP_FLAG_CONTEXT);
    c = c < 0 ? 0 : cap;
  }
  const int64_t t0 = (int64_t)split * p.split_len;
  const int64_t t1 = min(t0 + p.split_len, c);

  fused_append<D, 2>(p, r, hgi, HG, c, t0, t1);

  if (t0 >= t1) {
    for (int qi = 0; qi < Q; ++qi) {
      const int64_t rq = (int64_t)r * Q + qi;
      if (p.num_splits > 1) {
        for (int i = threadIdx.x; i < HG * Gr; i += blockDim.x)
          p.ws_lse[(rq * p.q_heads + hq0 + i) * p.num_splits + split] = -INFINITY;
      } else {
        __nv_bfloat16* o = static_cast<__nv_bfloat16*>(p.out) + (rq * p.q_heads + hq0) * D;
        for (int i = threadIdx.x; i < HG * Gr * D; i += blockDim.x) o[i] = __float2bfloat16_rn(0.f);
      }
    }
    return;
  }

  extern __shared__ __align__(1024) unsigned char smem_raw[];
  // the ring starts 1024-byte aligned (TMA's 128-byte swizzle repeats every
  // 1024 bytes of shared-memory address)
  unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const int stages = p.stages;
  const size_t stage_bytes = S::stage_bytes(HG);
  const size_t ring = S::ring_bytes(HG, stages, NC);
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + ring);
  uint64_t* empty_bar = full_bar + stages;
  volatile int* abort = reinterpret_cast<volatile int*>(empty_bar + stages);

  if (threadIdx.x == 0) {
    for (int i = 0; i < stages; ++i) {
      mbar_init(smem_u32(&full_bar[i]), 1);
      mbar_init(smem_u32(&empty_bar[i]), HG);  // one arrive per consumer warp
    }
    *abort = 0;
    fence_mbar_init();
  }
  __syncthreads();

  const int64_t nch = (t1 - t0 + C::CT - 1) / C::CT;
  // TMAP layout of a stage: [K | V] x [CT/B boxes] x [D/64 slabs of 64 dims]
  //                         x [HG heads] x [B token rows of 128 bytes]
  StageLayout<D, TMAP> L;
  L.BT = TMAP ? p.box_tokens : 1;
  L.slab_bytes = (uint32_t)L.BT * HG * 128;
  L.box_bytes = (uint32_t)(D / 64) * L.slab_bytes;
  L.RS = (uint32_t)S::row_stride(HG);
  L.hl = warp % HG;
  if (TMAP && (L.BT < 1 || L.BT > C::CT || C::CT % L.BT != 0)) {
    // a box must fit its stage; the host never launches otherwise
    if (threadIdx.x == 0) set_flag(p.err, NP_FLAG_CONFIG);
    return;
  }

  MmaWarp<D, G, TWO> W;
  W.mA = W.mB = -INFINITY;
  W.lA = W.lB = 0.f;

  if (warp == NC) {
    // ======================= producer warp
    const uint64_t pol = policy_evict_first();
    const int64_t nblk = (c + p.block_size - 1) / p.block_size;
    int64_t win = -1;
    int32_t my_id = 0;
    int64_t issued = 0;
    for (int64_t ch = 0; ch < nch; ++ch) {
      const int st = (int)(ch % stages);
      if (ch >= stages) {
        bool ok = mbar_wait(smem_u32(&empty_bar[st]), (uint32_t)((ch / stages - 1) & 1), abort);
        if (!__all_sync(FULL, ok)) break;
      }
      const int64_t cb = t0 + ch * C::CT;
      const int n = (int)min((int64_t)C::CT, t1 - cb);
      const uint32_t kdst = smem_u32(smem + st * stage_bytes);
      produce_chunk<D, TMAP>(p, L, r, hgi, HG, cb, n, nblk, kdst,
                             kdst + (uint32_t)(stage_bytes / 2), smem_u32(&full_bar[st]), pol,
                             win, my_id, lane);
      issued = ch + 1;
    }
    if (*abort) {  // never leave copies in flight (bounded)
      for (int64_t ch = max((int64_t)0, issued - stages); ch < issued; ++ch)
        mbar_wait_drain(smem_u32(&full_bar[ch % stages]), (uint32_t)((ch / stages) & 1));
    }
  } else {
    // ======================= consumer warp: kv head hl, chunks tw, tw+TW, ...
    const int tw = warp / HG;
    W.begin(p, r, hgi * HG + L.hl, c, lane);
    int st = tw % stages;                 // stage of chunk ch, and the parity of
    uint32_t fph = (tw / stages) & 1u;    // its full barrier's phase, kept incrementally
    for (int64_t ch = tw; ch < nch; ch += TW) {
      bool ok = mbar_wait(smem_u32(&full_bar[st]), fph, abort);
      if (!__all_sync(FULL, ok)) {
        set_flag(p.err, NP_FLAG_TIMEOUT);
        break;
      }
      const int64_t tch = t0 + ch * C::CT;  // position of the chunk's first token
      const int nvalid = (int)min((int64_t)C::CT, t1 - tch);
      const uint32_t kst = smem_u32(smem + st * stage_bytes);
      for (int sb = 0; sb < nvalid; sb += C::ST)
        W.template tile<TMAP>(L, kst, kst + (uint32_t)(stage_bytes / 2), sb, nvalid, tch,
                              p.qscale, lane);
      __syncwarp();  // every lane's reads of this stage are done
      if (lane == 0) mbar_arrive(smem_u32(&empty_bar[st]));
      for (st += TW; st >= stages; st -= stages) fph ^= 1u;
    }
    W.finish();
  }

  // ======================= epilogue: stage (m, l, O) per warp, merge, store
  __syncthreads();  // (A) ring no longer in use
  float* merge = reinterpret_cast<float*>(smem);
  if (warp < NC) {
    float* mg = merge + warp * kMmaRows * (D + 2);
    W.store_rows(mg, mg + kMmaRows, mg + 2 * kMmaRows, MR, lane);
  }
  __syncthreads();  // (B)
  if (warp >= NC || warp / HG != 0) return;
  split_write_rows<__nv_bfloat16, D>(p, merge, r, split, hgi * HG + warp, warp, HG, TW, Gr, lane);
}

}  // namespace npk
