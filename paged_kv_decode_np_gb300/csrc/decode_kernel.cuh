// decode_kernel.cuh -- the paged decode read, one kernel template per
// (storage type T, head_dim D, GQA group G).
//
// What it computes (per row r, query head h, kv head h / G): attention of
// the row's one query token over its whole history, the history gathered
// through the row's block table from a pool [num_blocks, block_size,
// kv_heads, head_dim] ("Day 17: paging under the sampling path", Diagram;
// "Day 25: the fused read dispatches to the kernel backend", What I added
// today).  The softmax is streamed: a running max m and sum l per head, the
// accumulator rescaled by 2^(m_old - m_new) whenever the max grows, so no
// full array of scores is ever built ("Day 60: the read becomes a choice", What
// I added today and Post angle; "Day 25", Why it matters: the streamed
// softmax sums the exponentials in another order, so results are close to,
// not bit-equal with, the exact softmax).
//
// Work decomposition (GB300 design, not from the pages):
//   grid  = (num_splits, rows, kv_heads / HG)
//   block = HG*TW consumer warps + 1 producer warp
// A CTA owns HG consecutive kv heads of one row and one split of its
// history.  Because the pool stores all kv heads of a token contiguously,
// the CTA's K (and V) bytes for a run of tokens in one block form ONE
// contiguous range when HG == kv_heads: the producer warp moves it with a
// single 1-D bulk TMA copy (cp.async.bulk) into a ring of shared-memory
// stages guarded by mbarriers.  Block ids are fetched 32 at a time by the
// producer's lanes and broadcast with shuffles.  Consumer warp (hl, tw)
// computes for kv head hl, all G query heads of its group (one K/V fetch
// serves the whole group), on chunks c with c % TW == tw.
//
// Inside a consumer warp, QK^T maps LD lanes across head_dim and LT = 32/LD
// lanes across tokens (partial dot products reduced with xor-shuffles over
// the LD lanes); PV maps LDV lanes across head_dim and LTV across tokens,
// with the probabilities passed through a small per-warp shared tile.
// Scores are kept in log2 units (q pre-multiplied by scale*log2(e)) so the
// exponentials are single ex2 instructions.
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
  // go to ws_o, each CTA's two merge descriptors to st_desc ([P][2][4]).
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

constexpr int floor_pow2(int x) {
  int p = 1;
  while (p * 2 <= x) p *= 2;
  return p;
}
constexpr int cmax(int a, int b) { return a > b ? a : b; }
constexpr int cmin(int a, int b) { return a < b ? a : b; }

template <typename T, int D, int G>
struct DecodeCfg {
  static constexpr int ES = sizeof(T);
  static constexpr int V16 = 16 / ES;  // elements per 16-byte vector
  // QK map: LD lanes across head_dim with DPL dims each (one or two 16-byte
  // vectors, the second half-way along the row so every quarter-warp reads
  // 128 contiguous bytes), LT lanes across tokens.  q stays in registers:
  // DPL * G <= 64 floats.
  static constexpr bool kBigOk = (2 * V16 <= D) && (2 * V16 * G <= 64);
  static constexpr bool kSmallOk = (D / V16) <= 32;
  static constexpr int DPL = (kBigOk || !kSmallOk) ? 2 * V16 : V16;
  static constexpr int LD = D / DPL;
  static constexpr int LT = 32 / LD;
  static constexpr int NVQ = DPL / V16;
  // PV map: LDV lanes across head_dim with DPV dims each, LTV across tokens.
  static constexpr int DPV = (D / 4 <= 32) ? 4 : D / 32;
  static constexpr int LDV = D / DPV;
  static constexpr int LTV = 32 / LDV;
  static constexpr int VPV = (DPV * ES <= 16) ? DPV : V16;
  static constexpr int NVPV = DPV / VPV;
  // Chunk = one pipeline stage, in tokens: about 64 KB of K+V at 8 kv heads.
  static constexpr int CT = cmin(32, cmax(cmax(8, cmax(LT, LTV)), 4096 / (D * ES)));
  // Softmax sub-tile: NPS passes of LT tokens, at most 32 score registers.
  static constexpr int NPS = cmin(floor_pow2(cmax(1, 32 / G)), CT / LT);
  static constexpr int ST = NPS * LT;
  static constexpr int GP = (G + 3) / 4 * 4;  // probability tile row stride
  static_assert(D % DPL == 0 && LD >= 1 && LD <= 32 && 32 % LD == 0, "QK map");
  static_assert(D % DPV == 0 && LDV >= 1 && LDV <= 32 && 32 % LDV == 0, "PV map");
  static_assert(CT % ST == 0 && CT % LTV == 0 && ST >= LT, "tiling");
};

// Shared-memory footprint of a launch (host and device agree on this).
template <typename T, int D, int G>
struct DecodeSmem {
  using C = DecodeCfg<T, D, G>;
  __host__ __device__ static constexpr size_t stage_bytes(int hg) {
    return 2ull * C::CT * hg * D * C::ES;
  }
  __host__ __device__ static constexpr size_t ptile_bytes(int warps) {
    return (size_t)warps * C::ST * C::GP * sizeof(float);
  }
  __host__ __device__ static constexpr size_t merge_bytes(int warps) {
    return (size_t)warps * G * (D + 2) * sizeof(float);
  }
  // ring (or merge scratch, which reuses it) | ptile | barriers | abort flag
  __host__ __device__ static constexpr size_t ring_bytes(int hg, int stages, int warps) {
    size_t ring = stage_bytes(hg) * stages;
    size_t m = merge_bytes(warps);
    return ((ring > m ? ring : m) + 127) / 128 * 128;
  }
  __host__ __device__ static constexpr size_t total(int hg, int stages, int warps) {
    return ring_bytes(hg, stages, warps) + ptile_bytes(warps) + 16ull * stages + 16;
  }
};

template <typename T, int D, int G>
__global__ void __launch_bounds__(kMaxThreads, 1)
    paged_decode_kernel(const __grid_constant__ DecodeParams p) {
  using C = DecodeCfg<T, D, G>;
  using S = DecodeSmem<T, D, G>;
  constexpr unsigned FULL = 0xffffffffu;

  const int split = blockIdx.x;
  const int r = blockIdx.y;
  const int hgi = blockIdx.z;
  const int HG = p.head_group;
  const int TW = p.token_warps;
  const int NC = HG * TW;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int hq0 = hgi * HG * G;  // first query head of this CTA

  // ---- the row's history length (clamped; flagged if out of range)
  const int64_t cap = (int64_t)p.max_blocks_per_row * p.block_size;
  int64_t c = p.context_lens[r];
  if (c < 0 || c > cap) {
    if (threadIdx.x == 0) set_flag(p.err, NP_FLAG_CONTEXT);
    c = c < 0 ? 0 : cap;
  }
  const int64_t t0 = (int64_t)split * p.split_len;
  const int64_t t1 = min(t0 + p.split_len, c);

  fused_append<D, C::ES>(p, r, hgi, HG, c, t0, t1);

  if (t0 >= t1) {  // nothing to read: an empty split / an empty row
    if (p.num_splits > 1) {
      for (int i = threadIdx.x; i < HG * G; i += blockDim.x)
        p.ws_lse[((int64_t)r * p.q_heads + hq0 + i) * p.num_splits + split] = -INFINITY;
    } else {
      T* o = static_cast<T*>(p.out) + ((int64_t)r * p.q_heads + hq0) * D;
      for (int i = threadIdx.x; i < HG * G * D; i += blockDim.x) o[i] = T(0.f);
    }
    return;
  }

  // ---- shared memory
  extern __shared__ __align__(128) unsigned char smem[];
  const int stages = p.stages;
  const size_t stage_bytes = S::stage_bytes(HG);
  const size_t ring = S::ring_bytes(HG, stages, NC);
  float* ptile_all = reinterpret_cast<float*>(smem + ring);
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + ring + S::ptile_bytes(NC));
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

  const int64_t nch = (t1 - t0 + C::CT - 1) / C::CT;  // chunks in this split
  const int row_elems = HG * D;                       // one token's row in a stage
  const uint32_t row_bytes = row_elems * C::ES;

  if (warp == NC) {
    // ======================= producer warp: block-table walk + bulk copies
    const uint64_t pol = policy_evict_first();
    const int64_t bs = p.block_size;
    const int64_t tab0 = (int64_t)r * p.max_blocks_per_row;
    const int64_t nblk = (c + bs - 1) / bs;  // table entries this row uses
    const bool whole = (HG == p.kv_heads);
    const int64_t pool_row = (int64_t)p.kv_heads * D * C::ES;  // bytes per slot
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
    // Never leave copies in flight: wait (bounded) for the newest chunk of
    // every stage.  In normal operation the consumers already did.
    if (*abort) {
      for (int64_t ch = max((int64_t)0, issued - stages); ch < issued; ++ch) {
        mbar_wait_drain(smem_u32(&full_bar[ch % stages]), (uint32_t)((ch / stages) & 1));
      }
    }
  } else {
    // ======================= consumer warp (kv head hl, token slot tw)
    const int hl = warp % HG;
    const int tw = warp / HG;
    const int kvh = hgi * HG + hl;
    const int dl = lane % C::LD, tl = lane / C::LD;
    const int dv = lane % C::LDV, tlv = lane / C::LDV;
    float* pt = ptile_all + warp * (C::ST * C::GP);

    // q for the G heads of this kv head, pre-scaled into log2 units
    float qf[G][C::DPL];
    {
      const T* qrow = static_cast<const T*>(p.q) + ((int64_t)r * p.q_heads + kvh * G) * D;
#pragma unroll
      for (int h = 0; h < G; ++h) {
#pragma unroll
        for (int j = 0; j < C::NVQ; ++j)
          Storage<T>::template load<C::V16>(qrow + h * D + j * (D / C::NVQ) + dl * C::V16,
                                            &qf[h][j * C::V16]);
#pragma unroll
        for (int e = 0; e < C::DPL; ++e) qf[h][e] *= p.qscale;
      }
    }

    float m[G], l[G], acc[G][C::DPV];
#pragma unroll
    for (int h = 0; h < G; ++h) {
      m[h] = -INFINITY;
      l[h] = 0.f;
#pragma unroll
      for (int e = 0; e < C::DPV; ++e) acc[h][e] = 0.f;
    }

    for (int64_t ch = tw; ch < nch; ch += TW) {
      const int st = (int)(ch % stages);
      bool ok = mbar_wait(smem_u32(&full_bar[st]), (uint32_t)((ch / stages) & 1), abort);
      if (!__all_sync(FULL, ok)) {
        set_flag(p.err, NP_FLAG_TIMEOUT);
        break;
      }
      const int nvalid = (int)min((int64_t)C::CT, t1 - (t0 + ch * C::CT));
      const T* Ks = reinterpret_cast<const T*>(smem + st * stage_bytes) + hl * D;
      const T* Vs = reinterpret_cast<const T*>(smem + st * stage_bytes + stage_bytes / 2) + hl * D;

      for (int sb = 0; sb < nvalid; sb += C::ST) {
        // ---- scores for ST tokens (NPS passes of LT tokens)
        float sc[C::NPS][G];
#pragma unroll
        for (int i = 0; i < C::NPS; ++i) {
          const T* krow = Ks + (sb + i * C::LT + tl) * row_elems;
          float kv[C::DPL];
#pragma unroll
          for (int j = 0; j < C::NVQ; ++j)
            Storage<T>::template load<C::V16>(krow + j * (D / C::NVQ) + dl * C::V16,
                                              &kv[j * C::V16]);
#pragma unroll
          for (int h = 0; h < G; ++h) {
            float a = 0.f;
#pragma unroll
            for (int e = 0; e < C::DPL; ++e) a = fmaf(qf[h][e], kv[e], a);
            sc[i][h] = a;
          }
        }
#pragma unroll
        for (int off = 1; off < C::LD; off <<= 1) {
#pragma unroll
          for (int i = 0; i < C::NPS; ++i)
#pragma unroll
            for (int h = 0; h < G; ++h) sc[i][h] += __shfl_xor_sync(FULL, sc[i][h], off);
        }
        // ---- online softmax update
        float alpha[G];
#pragma unroll
        for (int h = 0; h < G; ++h) {
          float mt = -INFINITY;
#pragma unroll
          for (int i = 0; i < C::NPS; ++i) {
            if (sb + i * C::LT + tl >= nvalid) sc[i][h] = -INFINITY;
            mt = fmaxf(mt, sc[i][h]);
          }
#pragma unroll
          for (int off = C::LD; off < 32; off <<= 1) mt = fmaxf(mt, __shfl_xor_sync(FULL, mt, off));
          const float mn = fmaxf(m[h], mt);
          alpha[h] = ex2(m[h] - mn);
          m[h] = mn;
          float ls = 0.f;
#pragma unroll
          for (int i = 0; i < C::NPS; ++i) {
            sc[i][h] = ex2(sc[i][h] - mn);
            ls += sc[i][h];
          }
          l[h] = fmaf(l[h], alpha[h], ls);
        }
        // ---- probabilities to the warp's tile (each value written once)
#pragma unroll
        for (int i = 0; i < C::NPS; ++i)
#pragma unroll
          for (int h = 0; h < G; ++h)
            if ((h % C::LD) == dl) pt[(i * C::LT + tl) * C::GP + h] = sc[i][h];
        __syncwarp();
        // ---- PV
#pragma unroll
        for (int h = 0; h < G; ++h)
#pragma unroll
          for (int e = 0; e < C::DPV; ++e) acc[h][e] *= alpha[h];
        const int nt = min(C::ST, nvalid - sb);
        for (int tt = tlv; tt < nt; tt += C::LTV) {
          float pv[C::GP];
#pragma unroll
          for (int k = 0; k < C::GP / 4; ++k) {
            const float4 v4 = *reinterpret_cast<const float4*>(pt + tt * C::GP + 4 * k);
            pv[4 * k] = v4.x; pv[4 * k + 1] = v4.y; pv[4 * k + 2] = v4.z; pv[4 * k + 3] = v4.w;
          }
          const T* vrow = Vs + (sb + tt) * row_elems;
          float vv[C::DPV];
#pragma unroll
          for (int j = 0; j < C::NVPV; ++j)
            Storage<T>::template load<C::VPV>(vrow + j * (D / C::NVPV) + dv * C::VPV,
                                              &vv[j * C::VPV]);
#pragma unroll
          for (int h = 0; h < G; ++h)
#pragma unroll
            for (int e = 0; e < C::DPV; ++e) acc[h][e] = fmaf(pv[h], vv[e], acc[h][e]);
        }
        __syncwarp();
      }
      __syncwarp();  // every lane's reads of this stage are done
      if (lane == 0) mbar_arrive(smem_u32(&empty_bar[st]));
    }

    // ---- combine the lanes' partial sums
#pragma unroll
    for (int h = 0; h < G; ++h) {
#pragma unroll
      for (int off = C::LD; off < 32; off <<= 1) l[h] += __shfl_xor_sync(FULL, l[h], off);
#pragma unroll
      for (int e = 0; e < C::DPV; ++e)
#pragma unroll
        for (int off = C::LDV; off < 32; off <<= 1)
          acc[h][e] += __shfl_xor_sync(FULL, acc[h][e], off);
    }

    // ---- several warps per kv head: merge through shared memory
    if (TW > 1) {
      __syncthreads();  // (A) every consumer is done with the ring
      float* mg = reinterpret_cast<float*>(smem) + warp * (G * (D + 2));
      if (lane == 0) {
#pragma unroll
        for (int h = 0; h < G; ++h) {
          mg[h] = m[h];
          mg[G + h] = l[h];
        }
      }
      if (tlv == 0) {
#pragma unroll
        for (int h = 0; h < G; ++h)
#pragma unroll
          for (int j = 0; j < C::NVPV; ++j)
#pragma unroll
            for (int e = 0; e < C::VPV; ++e)
              mg[2 * G + h * D + j * (D / C::NVPV) + dv * C::VPV + e] = acc[h][j * C::VPV + e];
      }
      __syncthreads();  // (B)
      if (tw != 0) return;
#pragma unroll
      for (int h = 0; h < G; ++h) {
        float mm = m[h];
        for (int w2 = 1; w2 < TW; ++w2) mm = fmaxf(mm, reinterpret_cast<float*>(smem)[(hl + w2 * HG) * (G * (D + 2)) + h]);
        const float a0 = (mm == -INFINITY) ? 0.f : ex2(m[h] - mm);
        float ll = l[h] * a0;
#pragma unroll
        for (int e = 0; e < C::DPV; ++e) acc[h][e] *= a0;
        for (int w2 = 1; w2 < TW; ++w2) {
          const float* o = reinterpret_cast<float*>(smem) + (hl + w2 * HG) * (G * (D + 2));
          const float a = (o[h] == -INFINITY) ? 0.f : ex2(o[h] - mm);
          ll = fmaf(o[G + h], a, ll);
#pragma unroll
          for (int j = 0; j < C::NVPV; ++j)
#pragma unroll
            for (int e = 0; e < C::VPV; ++e)
              acc[h][j * C::VPV + e] =
                  fmaf(o[2 * G + h * D + j * (D / C::NVPV) + dv * C::VPV + e], a,
                       acc[h][j * C::VPV + e]);
        }
        m[h] = mm;
        l[h] = ll;
      }
    }

    // ---- write the result (lanes of token-slot 0 own distinct dims)
    if (tlv == 0) {
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const int hq = kvh * G + h;
        const float inv = l[h] > 0.f ? 1.f / l[h] : 0.f;
        float o[C::DPV];
#pragma unroll
        for (int e = 0; e < C::DPV; ++e) o[e] = acc[h][e] * inv;
        if (p.num_splits == 1) {
          T* orow = static_cast<T*>(p.out) + ((int64_t)r * p.q_heads + hq) * D;
#pragma unroll
          for (int j = 0; j < C::NVPV; ++j)
            Storage<T>::template store<C::VPV>(orow + j * (D / C::NVPV) + dv * C::VPV,
                                               &o[j * C::VPV]);
        } else {
          const int64_t rs = ((int64_t)r * p.q_heads + hq) * p.num_splits + split;
          float* orow = p.ws_o + rs * D;
#pragma unroll
          for (int j = 0; j < C::NVPV; ++j)
#pragma unroll
            for (int k = 0; k < C::VPV; k += 4)
              Storage<float>::template store<4>(orow + j * (D / C::NVPV) + dv * C::VPV + k,
                                                &o[j * C::VPV + k]);
          if (dv == 0)
            p.ws_lse[rs] = l[h] > 0.f ? m[h] * 0.69314718055994531f + logf(l[h]) : -INFINITY;
        }
      }
    }
    return;
  }

  // producer warp: take part in the merge barriers of the consumers
  if (TW > 1) {
    __syncthreads();  // (A)
    __syncthreads();  // (B)
  }
}

}  // namespace npk
