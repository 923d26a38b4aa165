// decode_fma.cuh -- the fp32 consumer warp of the balanced read: one kv
// head, its G query heads (times the row's query tokens), full fp32 products
// on the FMA pipes.
//
// What it computes is the read of decode_kernel.cuh (scores q.K in log2
// units, a running max and sum per head, the accumulator rescaled when the
// max grows).  The work layout is chosen for instruction count and
// independent chains on the FMA pipes:
//   * QK: lane (dl, tg) owns head_dim slice dl (DPL dims) of the chunk's
//     token group tg (NT tokens); it forms the partial dot products of all
//     NT tokens x G heads -- NT*GP independent FMA chains of DPL terms.
//   * The LD lanes of a token group sum those partials with a shuffle
//     reduce-scatter (each level keeps half of the values and adds the
//     partner's other half), so every score is finished by one lane with
//     NT*GP - 1 shuffles in all rather than log2(LD) per score.
//   * Softmax: finished scores go through a small per-warp tile into a
//     (token, head) lane layout; lanes of one head reduce the chunk max and
//     sum with xor-shuffles, write the probabilities and each head's
//     rescale factor back to the tile.
//   * PV: lane (dl, tg) again owns head_dim slice dl and accumulates
//     p[t][h] * V[t][dl] over its token group; token groups are summed at the
//     end.
// Rows: with one query token per row, the G heads (padded to a power of two);
// with several (MQ), rows qi*G + h for query token qi and head h, up to 8,
// each masked to the positions at or before its own (c - Q + qi), as in the
// tensor-core warp.  G = 0 (with MQ): the group is read at run time, for
// groups outside the compiled set.
// Stage layout (written by the producer's bulk copies): K rows [token][hg kv
// heads][D] fp32, then V rows the same.
#pragma once

#include "decode_kernel.cuh"
#include "decode_mma.cuh"  // kMmaRows, split_write_rows

namespace npk {

template <int D, int G, bool MQ = false>
struct FmaCfg {
  static constexpr int LD = D / 4 < 32 ? D / 4 : 32;  // lanes across head_dim
  static constexpr int DPL = D / LD;                   // dims per lane: 4 (8 at D = 256)
  static constexpr int LT = 32 / LD;                   // token groups
  static constexpr int CT = 1024 / D;                  // tokens per stage: 64 KB of K+V at 8 heads
  static constexpr int NT = CT / LT;                   // tokens per lane per chunk
  static constexpr int NR = MQ ? 8 : G;                // rows computed
  static constexpr int GP = MQ ? 8 : (G <= 1 ? 1 : G <= 2 ? 2 : G <= 4 ? 4 : 8);  // padded rows
  static constexpr int NV = NT * GP;                   // partial scores per lane
  static constexpr int LOG_LD = LD >= 32 ? 5 : LD >= 16 ? 4 : LD >= 8 ? 3 : LD >= 4 ? 2 : 1;
  static constexpr int NE = (CT * GP + 31) / 32;       // tile entries per lane in the softmax
  static constexpr int TILE = CT * GP + 8;             // floats per warp: p[CT][GP], alpha[GP]
  static_assert(D % 16 == 0 && D <= 256, "fp32 consumer: head_dim 16..256");
  static_assert(DPL % 4 == 0 && 32 % LD == 0 && CT % LT == 0 && NT >= 1, "fp32 layout");
  static_assert(G <= 8, "fp32 balanced read: at most 8 query heads per kv head");
  static_assert(G > 0 || MQ, "a group read at run time takes the 8-row layout");
};

template <int D, int G, bool MQ = false>
struct FmaWarp {
  using C = FmaCfg<D, G, MQ>;
  static constexpr int NR = C::NR;
  float q[NR][C::DPL];    // this lane's head_dim slice of each row's q (log2 units)
  float acc[NR][C::DPL];  // unnormalised output slice
  float m, l;             // running max and sum of row (lane % GP)
  int32_t lim;            // last position row (lane % GP) may see (-1: a padding row);
                          // positions fit int32 on the balanced read
  int gr;                 // query heads per kv head (G, or q_heads/kv_heads when G = 0)

  __device__ __forceinline__ void begin(const DecodeParams& p, int64_t r, int kvh, int64_t c,
                                        int lane) {
    gr = G > 0 ? G : p.q_heads / p.kv_heads;
    const int Q = p.query_len, MR = gr * Q;
    const int dl = lane % C::LD;
#pragma unroll
    for (int row = 0; row < NR; ++row) {
      const int qi = row / gr, h = row - (row / gr) * gr;
      if (row < MR) {
        const float* qr = static_cast<const float*>(p.q) +
                          ((r * Q + qi) * p.q_heads + (int64_t)kvh * gr + h) * D;
        Storage<float>::template load<C::DPL>(qr + dl * C::DPL, q[row]);
      }
#pragma unroll
      for (int e = 0; e < C::DPL; ++e) {
        q[row][e] = row < MR ? q[row][e] * p.qscale : 0.f;
        acc[row][e] = 0.f;
      }
    }
    const int rme = lane % C::GP;
    lim = rme < MR ? (int32_t)(c - Q + rme / gr) : -1;
    m = -INFINITY;
    l = 0.f;
  }

  // One staged chunk: K rows at ks, V rows at vs ([token][hg][D] floats, this
  // warp's kv head hl), its first token at position cb and the first nvalid
  // tokens valid; tile = the warp's scratch of C::TILE floats.
  __device__ __forceinline__ void consume(const float* ks, const float* vs, int hl, int hg,
                                          int nvalid, int64_t cb, float* tile, int lane) {
    constexpr unsigned FULL = 0xffffffffu;
    constexpr int GP = C::GP, NT = C::NT, DPL = C::DPL;
    const int dl = lane % C::LD, tg = lane / C::LD;
    const int t0 = tg * NT;  // this lane's first token of the chunk
    const int rowf = hg * D;  // floats per token row of a stage

    // ---- partial scores x[j*GP + h] over this lane's head_dim slice
    float x[C::NV];
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      float kv[DPL];
      Storage<float>::template load<DPL>(ks + (t0 + j) * rowf + hl * D + dl * DPL, kv);
#pragma unroll
      for (int h = 0; h < GP; ++h) {
        float a = 0.f;
        if (h < NR) {
#pragma unroll
          for (int e = 0; e < DPL; ++e) a = fmaf(q[h][e], kv[e], a);
        }
        x[j * GP + h] = a;
      }
    }
    // ---- reduce-scatter over the LD lanes of the token group
    int base = 0;  // index of x[0] after the scatter levels
#pragma unroll
    for (int k = 0; k < C::LOG_LD; ++k) {
      const int msk = 1 << k;
      const int n = C::NV >> k;  // values still held
      if (n >= 2) {
        const bool up = (lane & msk) != 0;
        const int half = n / 2;
#pragma unroll
        for (int i = 0; i < half; ++i) {
          const float send = up ? x[i] : x[i + half];
          const float keep = up ? x[i + half] : x[i];
          x[i] = keep + __shfl_xor_sync(FULL, send, msk);
        }
        if (up) base += half;
      } else {
        x[0] += __shfl_xor_sync(FULL, x[0], msk);
      }
    }
    constexpr int NF = C::NV >= C::LD ? C::NV / C::LD : 1;  // finished scores per lane
    constexpr int SCAT = C::NV >= C::LD ? C::LOG_LD
                         : (C::NV >= 32 ? 5 : C::NV >= 16 ? 4 : C::NV >= 8 ? 3
                            : C::NV >= 4 ? 2 : C::NV >= 2 ? 1 : 0);
    if ((dl >> SCAT) == 0) {  // one writer per finished score
#pragma unroll
      for (int i = 0; i < NF; ++i) tile[t0 * GP + base + i] = x[i];
    }
    __syncwarp();

    // ---- softmax in the (token, row) layout: entry e = t*GP + row; every
    // entry of this lane belongs to row lane % GP, which may see positions
    // up to lim
    float s[C::NE];
    float mt = -INFINITY;
#pragma unroll
    for (int k = 0; k < C::NE; ++k) {
      const int e = lane + 32 * k;
      const bool ok = e < C::CT * GP && e / GP < nvalid && (int32_t)cb + e / GP <= lim;
      s[k] = ok ? tile[e] : -INFINITY;
      mt = fmaxf(mt, s[k]);
    }
#pragma unroll
    for (int o = GP; o < 32; o <<= 1) mt = fmaxf(mt, __shfl_xor_sync(FULL, mt, o));
    const float mn = fmaxf(m, mt);
    const float msub = mn == -INFINITY ? 0.f : mn;
    const float alpha = ex2(m - msub);  // m = -inf: 0 (nothing accumulated yet)
    float ls = 0.f;
#pragma unroll
    for (int k = 0; k < C::NE; ++k) {
      s[k] = ex2(s[k] - msub);  // -inf: 0
      ls += s[k];
    }
#pragma unroll
    for (int o = GP; o < 32; o <<= 1) ls += __shfl_xor_sync(FULL, ls, o);
    l = fmaf(l, alpha, ls);
    m = mn;
    __syncwarp();  // every score has been read
#pragma unroll
    for (int k = 0; k < C::NE; ++k) {
      const int e = lane + 32 * k;
      if (e < C::CT * GP) tile[e] = s[k];
    }
    if (lane < GP) tile[C::CT * GP + lane] = alpha;
    __syncwarp();

    // ---- PV over this lane's tokens and head_dim slice
    float al[GP];
#pragma unroll
    for (int h = 0; h < GP; ++h) al[h] = tile[C::CT * GP + h];
#pragma unroll
    for (int h = 0; h < NR; ++h)
#pragma unroll
      for (int e = 0; e < DPL; ++e) acc[h][e] *= al[h];
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      const int t = t0 + j;
      if (t < nvalid) {
        float pj[GP], vv[DPL];
#pragma unroll
        for (int h = 0; h < GP; ++h) pj[h] = tile[t * GP + h];
        Storage<float>::template load<DPL>(vs + t * rowf + hl * D + dl * DPL, vv);
#pragma unroll
        for (int h = 0; h < NR; ++h)
#pragma unroll
          for (int e = 0; e < DPL; ++e) acc[h][e] = fmaf(pj[h], vv[e], acc[h][e]);
      }
    }
    __syncwarp();  // the tile is free for the next chunk
  }

  // token groups' partial outputs summed (lanes tg == 0 end with the result)
  __device__ __forceinline__ void finish() {
    constexpr unsigned FULL = 0xffffffffu;
#pragma unroll
    for (int o = C::LD; o < 32; o <<= 1)
#pragma unroll
      for (int h = 0; h < NR; ++h)
#pragma unroll
        for (int e = 0; e < C::DPL; ++e) acc[h][e] += __shfl_xor_sync(FULL, acc[h][e], o);
  }

  // The whole row's normalised output: row qi*G + h to out[r, qi, kvh*G + h].
  __device__ __forceinline__ void store_out(const DecodeParams& p, int64_t r, int kvh,
                                            int lane) const {
    constexpr unsigned FULL = 0xffffffffu;
    const int Q = p.query_len, MR = gr * Q;
    const int dl = lane % C::LD;
#pragma unroll
    for (int row = 0; row < NR; ++row) {
      const float lh = __shfl_sync(FULL, l, row);  // lane `row` holds that row's sum
      const float inv = lh > 0.f ? 1.f / lh : 0.f;
      float v[C::DPL];
#pragma unroll
      for (int e = 0; e < C::DPL; ++e) v[e] = acc[row][e] * inv;
      const int qi = row / gr, h = row - (row / gr) * gr;
      float* o = static_cast<float*>(p.out) + ((r * Q + qi) * p.q_heads + (int64_t)kvh * gr + h) * D;
      if (lane < C::LD && row < MR) Storage<float>::template store<C::DPL>(o + dl * C::DPL, v);
    }
  }

  // Unnormalised rows into a [16 rows][D] fp32 array plus m and l ([16]
  // each) through the store st, as the merges read them; rows >= MR are
  // skipped.
  template <typename St = PlainStore>
  __device__ __forceinline__ void store_rows(float* m_out, float* l_out, float* o_out, int MR,
                                             int lane, St st = St()) const {
    const int dl = lane % C::LD;
    if (lane < MR && lane < NR) {
      st(&m_out[lane], m);
      st(&l_out[lane], l);
    }
    if (lane < C::LD) {
#pragma unroll
      for (int row = 0; row < NR; ++row)
        if (row < MR) {
#pragma unroll
          for (int e = 0; e < C::DPL; e += 4) st.v4(o_out + row * D + dl * C::DPL + e, &acc[row][e]);
        }
    }
  }
};


// ------------------------------------------------------------------------
// The split grid on fp32 pools: grid (num_splits, rows, kv_heads / HG),
// HG*TW consumer warps (FmaWarp, one kv head each; the TW warps of a head
// take alternate chunks) + 1 producer warp.  A CTA reads tokens
// [split*split_len, +split_len) of its row for HG kv heads; the producer
// walks the row's block table (32 entries per load, broadcast by shuffles)
// and stages chunks of CT token rows [token][HG heads][D] fp32 with 1-D bulk
// copies -- one per run of tokens inside a block when the pool holds just
// the CTA's HG kv heads (a contiguous range), else one per token row.  The
// TW warps of a head merge their states at the end (split_write_rows) and
// write the rows' output, or this split's partials for the reduce.

// Shared memory: ring (after the read: the warps' (m, l, O) rows for the
// merge) | per-warp consumer tiles | full, empty barriers | abort flag.
template <int D, int G, bool MQ>
struct FmaSplitSmem {
  using C = FmaCfg<D, G, MQ>;
  __host__ __device__ static constexpr size_t stage_bytes(int hg) {
    return 2ull * C::CT * hg * D * sizeof(float);
  }
  __host__ __device__ static constexpr size_t ring_bytes(int hg, int stages, int warps) {
    const size_t ring = stage_bytes(hg) * stages;
    const size_t m = (size_t)warps * kMmaRows * (D + 2) * sizeof(float);
    return ((ring > m ? ring : m) + 127) / 128 * 128;
  }
  __host__ __device__ static constexpr size_t tiles_bytes(int warps) {
    return (size_t)warps * C::TILE * sizeof(float);
  }
  __host__ __device__ static constexpr size_t total(int hg, int stages, int warps) {
    return ring_bytes(hg, stages, warps) + tiles_bytes(warps) + 16ull * stages + 16;
  }
};

template <int D, int G, bool MQ>
__global__ void __launch_bounds__(kMaxThreads, 1)
    paged_decode_fma_kernel(const __grid_constant__ DecodeParams p) {
  using C = FmaCfg<D, G, MQ>;
  using S = FmaSplitSmem<D, G, MQ>;
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
  const int MR = Gr * Q;  // (query token, head) rows, <= 8

  const int64_t cap = (int64_t)p.max_blocks_per_row * p.block_size;
  int64_t c = p.context_lens[r];
  if (c < 0 || c > cap) {
    if (threadIdx.x == 0) set_flag(p.err, NP_FLAG_CONTEXT);
    c = c < 0 ? 0 : cap;
  }
  const int64_t t0 = (int64_t)split * p.split_len;
  const int64_t t1 = min(t0 + p.split_len, c);

  fused_append<D, 4>(p, r, hgi, HG, c, t0, t1);

  if (t0 >= t1) {  // nothing to read: an empty split / an empty row
    for (int qi = 0; qi < Q; ++qi) {
      const int64_t rq = (int64_t)r * Q + qi;
      if (p.num_splits > 1) {
        for (int i = threadIdx.x; i < HG * Gr; i += blockDim.x)
          p.ws_lse[(rq * p.q_heads + hq0 + i) * p.num_splits + split] = -INFINITY;
      } else {
        float* o = static_cast<float*>(p.out) + (rq * p.q_heads + hq0) * D;
        for (int i = threadIdx.x; i < HG * Gr * D; i += blockDim.x) o[i] = 0.f;
      }
    }
    return;
  }

  extern __shared__ __align__(128) unsigned char smem[];
  const int stages = p.stages;
  const size_t stage_bytes = S::stage_bytes(HG);
  const size_t ring = S::ring_bytes(HG, stages, NC);
  float* tiles = reinterpret_cast<float*>(smem + ring);
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + ring + S::tiles_bytes(NC));
  uint64_t* empty_bar = full_bar + stages;
  volatile int* abort = reinterpret_cast<volatile int*>(empty_bar + stages);

  if (threadIdx.x == 0) {
    for (int i = 0; i < stages; ++i) {
      mbar_init(smem_u32(&full_bar[i]), 1);
      mbar_init(smem_u32(&empty_bar[i]), HG);  // one arrive per consumer warp of a chunk
    }
    *abort = 0;
    fence_mbar_init();
  }
  __syncthreads();

  const int64_t nch = (t1 - t0 + C::CT - 1) / C::CT;  // chunks in this split
  const uint32_t row_bytes = (uint32_t)HG * D * sizeof(float);  // a token's row in a stage
  FmaWarp<D, G, MQ> W;

  if (warp == NC) {
    // ======================= producer warp: block-table walk + bulk copies
    const uint64_t pol = policy_evict_first();
    const int64_t bs = p.block_size;
    const int64_t tab0 = (int64_t)r * p.max_blocks_per_row;
    const int64_t nblk = (c + bs - 1) / bs;  // table entries this row uses
    const bool whole = (HG == p.kv_heads);
    const int64_t pool_row = (int64_t)p.kv_heads * D * sizeof(float);  // bytes per slot
    const char* kpool = static_cast<const char*>(p.k_pool) + (int64_t)hgi * row_bytes;
    const char* vpool = static_cast<const char*>(p.v_pool) + (int64_t)hgi * row_bytes;
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
      const int64_t ce = min(cb + (int64_t)C::CT, t1);
      const uint32_t fb = smem_u32(&full_bar[st]);
      const uint32_t kdst = smem_u32(smem + st * stage_bytes);
      const uint32_t vdst = kdst + (uint32_t)(stage_bytes / 2);
      if (lane == 0) mbar_arrive_expect_tx(fb, 2u * (uint32_t)(ce - cb) * row_bytes);
      for (int64_t t = cb; t < ce;) {
        const int64_t j = t / bs;
        const int64_t off = t - j * bs;
        const int64_t n = min(bs - off, ce - t);
        if (win < 0 || j >= win + 32) {
          win = j;
          const int64_t jj = j + lane;
          my_id = jj < nblk ? p.block_tables[tab0 + jj] : 0;
        }
        int64_t b = __shfl_sync(FULL, my_id, (int)(j - win));
        if (b < 0 || b >= p.num_blocks) {
          if (lane == 0) set_flag(p.err, NP_FLAG_BLOCK_ID);
          b = 0;
        }
        const int64_t slot = b * bs + off;
        const uint32_t so = (uint32_t)(t - cb) * row_bytes;
        if (whole) {
          if (lane == 0) {
            bulk_g2s(kdst + so, kpool + slot * pool_row, (uint32_t)n * row_bytes, fb, pol);
            bulk_g2s(vdst + so, vpool + slot * pool_row, (uint32_t)n * row_bytes, fb, pol);
          }
        } else {
          for (int64_t i = lane; i < n; i += 32) {
            bulk_g2s(kdst + so + (uint32_t)i * row_bytes, kpool + (slot + i) * pool_row,
                     row_bytes, fb, pol);
            bulk_g2s(vdst + so + (uint32_t)i * row_bytes, vpool + (slot + i) * pool_row,
                     row_bytes, fb, pol);
          }
        }
        t += n;
      }
      issued = ch + 1;
    }
    if (*abort) {  // never leave copies in flight (bounded)
      for (int64_t ch = max((int64_t)0, issued - stages); ch < issued; ++ch)
        mbar_wait_drain(smem_u32(&full_bar[ch % stages]), (uint32_t)((ch / stages) & 1));
    }
  } else {
    // ======================= consumer warp: kv head hl, chunks tw, tw+TW, ...
    const int hl = warp % HG;
    const int tw = warp / HG;
    float* tile = tiles + (size_t)warp * C::TILE;
    W.begin(p, r, hgi * HG + hl, c, lane);
    for (int64_t ch = tw; ch < nch; ch += TW) {
      const int st = (int)(ch % stages);
      bool ok = mbar_wait(smem_u32(&full_bar[st]), (uint32_t)((ch / stages) & 1), abort);
      if (!__all_sync(FULL, ok)) {
        set_flag(p.err, NP_FLAG_TIMEOUT);
        break;
      }
      const int64_t tch = t0 + ch * C::CT;  // position of the chunk's first token
      const int nvalid = (int)min((int64_t)C::CT, t1 - tch);
      const float* ks = reinterpret_cast<const float*>(smem + st * stage_bytes);
      W.consume(ks, ks + stage_bytes / 8, hl, HG, nvalid, tch, tile, lane);
      __syncwarp();  // every lane's reads of this stage are done
      if (lane == 0) mbar_arrive(smem_u32(&empty_bar[st]));
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
  split_write_rows<float, D>(p, merge, r, split, hgi * HG + warp, warp, HG, TW, Gr, lane);
}

}  // namespace npk
