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

#ifndef NPK_MMA_CT
#define NPK_MMA_CT 16  // tokens per pipeline stage for head_dim >= 64
#endif
#ifndef NPK_MMA_MIN_BLOCKS
#define NPK_MMA_MIN_BLOCKS 1  // resident CTAs per SM the register budget targets
#endif

template <int D, int G, bool TMAP>
struct MmaCfg {
  static constexpr int KS = D / 16;  // mma k-steps over head_dim (QK), m-tiles (PV)
  static constexpr int ST = 16;      // tokens per softmax tile
  static constexpr int CT = D >= 64 ? NPK_MMA_CT : 32;  // tokens per stage
  // CT < ST is allowed: the tile's rows past the chunk are masked and their
  // shared-memory reads are redirected to the tile's first row.
  static_assert(D % 16 == 0 && G >= 1 && G <= 8, "shape");
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
    return (size_t)warps * G * (D + 2) * sizeof(float);
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

template <int D, int G, bool TMAP>
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
  const int hq0 = hgi * HG * G;

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
    if (p.num_splits > 1) {
      for (int i = threadIdx.x; i < HG * G; i += blockDim.x)
        p.ws_lse[((int64_t)r * p.q_heads + hq0 + i) * p.num_splits + split] = -INFINITY;
    } else {
      __nv_bfloat16* o = static_cast<__nv_bfloat16*>(p.out) + ((int64_t)r * p.q_heads + hq0) * D;
      for (int i = threadIdx.x; i < HG * G * D; i += blockDim.x) o[i] = __float2bfloat16_rn(0.f);
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
  const uint32_t row_bytes = (uint32_t)HG * D * 2;  // one token, HG kv heads
  // TMAP layout of a stage: [K | V] x [D/64 slabs of 64 dims] x [CT/B boxes]
  //                         x [HG heads] x [B token rows of 128 bytes]
  const int BT = TMAP ? p.box_tokens : 1;
  const uint32_t half_bytes = (uint32_t)C::CT * HG * 128;  // one 64-dim slab of a chunk
  const uint32_t box_bytes = (uint32_t)BT * HG * 128;      // one box within a slab
  const uint32_t RS = (uint32_t)S::row_stride(HG);         // padded layout

  float m_run = -INFINITY, l_run = 0.f;
  float o[C::KS][4];  // O^T fragments: rows d = 16*mi + lane/4 (+8), cols h = 2*(lane%4) (+1)

  if (warp == NC) {
    // ======================= producer warp
    const uint64_t pol = policy_evict_first();
    const int64_t bs = p.block_size;
    const int64_t tab0 = (int64_t)r * p.max_blocks_per_row;
    const int64_t nblk = (c + bs - 1) / bs;
    const int64_t pool_row = (int64_t)p.kv_heads * D * 2;
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
      const int n = (int)min((int64_t)C::CT, t1 - cb);
      const uint32_t fb = smem_u32(&full_bar[st]);
      const uint32_t kdst = smem_u32(smem + st * stage_bytes);
      const uint32_t vdst = kdst + (uint32_t)(stage_bytes / 2);
      const int64_t jfirst = cb / bs;
      const int64_t jlast = (cb + n - 1) / bs;
      if (win < 0 || jlast >= win + 32) {
        win = jfirst;
        const int64_t jj = win + lane;
        my_id = jj < nblk ? p.block_tables[tab0 + jj] : 0;
      }
      if constexpr (TMAP) {
        // boxes of BT tokens; each lies inside one block (BT divides the block
        // size and the chunk start) and is copied whole (rows past the
        // history are masked by the consumers)
        const int nbox = (n + BT - 1) / BT;
        if (lane == 0) mbar_arrive_expect_tx(fb, 2u * (D / 64) * nbox * box_bytes);
        const int items = nbox * (D / 64) * 2;  // (box, slab, K|V)
        const int rounds = (items + 31) / 32;
        for (int rd = 0; rd < rounds; ++rd) {
          const int it = rd * 32 + lane;
          const int bx = (it < items ? it : 0) / ((D / 64) * 2);
          const int64_t t = cb + (int64_t)bx * BT;
          const int64_t j = t / bs;
          int64_t b = __shfl_sync(FULL, my_id, (int)(j - win));
          if (it < items) {
            const int slab = (it >> 1) % (D / 64);
            const bool isv = (it & 1) != 0;
            if (b < 0 || b >= p.num_blocks) {
              set_flag(p.err, NP_FLAG_BLOCK_ID);
              b = 0;
            }
            const int64_t slot = b * bs + (t - j * bs);
            const uint32_t dst = (isv ? vdst : kdst) + slab * half_bytes + bx * box_bytes;
            tma_load_3d(dst, isv ? &p.tm_v : &p.tm_k, slab * 64, (int32_t)slot, hgi * HG, fb,
                        pol);
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
          bulk_g2s(kdst + lane * RS, kpool + slot * pool_row, row_bytes, fb, pol);
          bulk_g2s(vdst + lane * RS, vpool + slot * pool_row, row_bytes, fb, pol);
        }
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
    const int kvh = hgi * HG + hl;
    const int g4 = lane >> 2;  // fragment row group
    const int c4 = lane & 3;   // fragment column pair

    // q as mma A fragments (rows = query heads of this group; rows >= G zero)
    uint32_t qa0[C::KS], qa2[C::KS];
    {
      const __nv_bfloat16* qrow =
          static_cast<const __nv_bfloat16*>(p.q) + ((int64_t)r * p.q_heads + kvh * G) * D;
#pragma unroll
      for (int ks = 0; ks < C::KS; ++ks) {
        if (g4 < G) {
          qa0[ks] = *reinterpret_cast<const uint32_t*>(qrow + g4 * D + 16 * ks + 2 * c4);
          qa2[ks] = *reinterpret_cast<const uint32_t*>(qrow + g4 * D + 16 * ks + 8 + 2 * c4);
        } else {
          qa0[ks] = 0u;
          qa2[ks] = 0u;
        }
      }
    }
#pragma unroll
    for (int mi = 0; mi < C::KS; ++mi)
#pragma unroll
      for (int e = 0; e < 4; ++e) o[mi][e] = 0.f;

    // ldmatrix lane addressing: matrix (lane/8) covers tokens 8*(lane/16) +
    // (0..7) and the 8-dim column chunk (lane/8)%2 of a 16-dim step; the same
    // pattern serves K (B of QK) and V (A of PV, transposed load)
    const int ld_tok = ((lane >> 4) << 3) + (lane & 7);
    const int ld_c = (lane >> 3) & 1;

    for (int64_t ch = tw; ch < nch; ch += TW) {
      const int st = (int)(ch % stages);
      bool ok = mbar_wait(smem_u32(&full_bar[st]), (uint32_t)((ch / stages) & 1), abort);
      if (!__all_sync(FULL, ok)) {
        set_flag(p.err, NP_FLAG_TIMEOUT);
        break;
      }
      const int nvalid = (int)min((int64_t)C::CT, t1 - (t0 + ch * C::CT));
      const uint32_t kst = smem_u32(smem + st * stage_bytes);
      const uint32_t vst = kst + (uint32_t)(stage_bytes / 2);

      for (int sb = 0; sb < nvalid; sb += C::ST) {
        // rows past the valid tokens read row sb instead (finite data; their
        // probabilities are exactly 0)
        const int tok = (sb + ld_tok < nvalid) ? sb + ld_tok : sb;
        // this lane's row within a slab, and its swizzle
        uint32_t row_off, swz = 0;
        if constexpr (TMAP) {
          const int bx = tok / BT, tr = tok - bx * BT;
          row_off = bx * box_bytes + (hl * BT + tr) * 128;
          swz = (row_off >> 7) & 7;
        } else {
          row_off = tok * RS + hl * D * 2;
        }
        // address of this lane's 16-byte chunk of dims [16*ks + 8*ld_c, +8)
        auto chunk_addr = [&](uint32_t base, int ks) -> uint32_t {
          if constexpr (TMAP) {
            const uint32_t cidx = ((2 * ks) & 7) + ld_c;  // chunk within the 128-byte row
            return base + (ks >> 2) * half_bytes + row_off + ((cidx ^ swz) << 4);
          } else {
            return base + row_off + ks * 32 + ld_c * 16;
          }
        };
        // ---- S^T = q K^T for 16 tokens (two n-tiles of 8)
        float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int ks = 0; ks < C::KS; ++ks) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4(chunk_addr(kst, ks), b0, b1, b2, b3);
          mma_bf16(s0, qa0[ks], 0u, qa2[ks], 0u, b0, b1);
          mma_bf16(s1, qa0[ks], 0u, qa2[ks], 0u, b2, b3);
        }
        // ---- online softmax (this lane: head g4, tokens 2*c4+{0,1} and 8+2*c4+{0,1})
        float sc[4] = {s0[0] * p.qscale, s0[1] * p.qscale, s1[0] * p.qscale, s1[1] * p.qscale};
        const int tb = sb + 2 * c4;
        if (tb >= nvalid) sc[0] = -INFINITY;
        if (tb + 1 >= nvalid) sc[1] = -INFINITY;
        if (tb + 8 >= nvalid) sc[2] = -INFINITY;
        if (tb + 9 >= nvalid) sc[3] = -INFINITY;
        float mt = fmaxf(fmaxf(sc[0], sc[1]), fmaxf(sc[2], sc[3]));
        mt = fmaxf(mt, __shfl_xor_sync(FULL, mt, 1));
        mt = fmaxf(mt, __shfl_xor_sync(FULL, mt, 2));
        const float mn = fmaxf(m_run, mt);
        const float alpha = ex2(m_run - mn);
        m_run = mn;
        float pr[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) pr[e] = ex2(sc[e] - mn);
        l_run = fmaf(l_run, alpha, (pr[0] + pr[1]) + (pr[2] + pr[3]));
        const uint32_t pb0 = pack_bf16(pr[0], pr[1]);
        const uint32_t pb1 = pack_bf16(pr[2], pr[3]);
        // ---- rescale O^T columns (heads 2*c4, 2*c4+1) when some max moved
        if (__any_sync(FULL, alpha != 1.f)) {
          const float a_lo = __shfl_sync(FULL, alpha, 8 * c4);
          const float a_hi = __shfl_sync(FULL, alpha, 8 * c4 + 4);
#pragma unroll
          for (int mi = 0; mi < C::KS; ++mi) {
            o[mi][0] *= a_lo;
            o[mi][1] *= a_hi;
            o[mi][2] *= a_lo;
            o[mi][3] *= a_hi;
          }
        }
        // ---- O^T += V^T P^T
#pragma unroll
        for (int mi = 0; mi < C::KS; ++mi) {
          uint32_t a0, a1, a2, a3;
          ldsm_x4_t(chunk_addr(vst, mi), a0, a1, a2, a3);
          mma_bf16(o[mi], a0, a1, a2, a3, pb0, pb1);
        }
      }
      __syncwarp();  // every lane's reads of this stage are done
      if (lane == 0) mbar_arrive(smem_u32(&empty_bar[st]));
    }
    // the head's sum over its 4 lanes
    l_run += __shfl_xor_sync(FULL, l_run, 1);
    l_run += __shfl_xor_sync(FULL, l_run, 2);
  }

  // ======================= epilogue: stage (m, l, O) per warp, merge, store
  __syncthreads();  // (A) ring no longer in use
  float* merge = reinterpret_cast<float*>(smem);
  const int stride_w = G * (D + 2);
  if (warp < NC) {
    float* mg = merge + warp * stride_w;
    if ((lane & 3) == 0 && (lane >> 2) < G) {
      mg[lane >> 2] = m_run;
      mg[G + (lane >> 2)] = l_run;
    }
    const int h0 = 2 * (lane & 3);
#pragma unroll
    for (int mi = 0; mi < C::KS; ++mi) {
      const int d = 16 * mi + (lane >> 2);
      if (h0 < G) {
        mg[2 * G + h0 * D + d] = o[mi][0];
        mg[2 * G + h0 * D + d + 8] = o[mi][2];
      }
      if (h0 + 1 < G) {
        mg[2 * G + (h0 + 1) * D + d] = o[mi][1];
        mg[2 * G + (h0 + 1) * D + d + 8] = o[mi][3];
      }
    }
  }
  __syncthreads();  // (B)
  if (warp >= NC || warp / HG != 0) return;
  const int hl = warp;  // tw == 0
  const int kvh = hgi * HG + hl;
  constexpr int DL = D >= 32 ? D / 32 : 1;  // dims per lane
  const int d0 = lane * DL;
  for (int h = 0; h < G; ++h) {
    float mm = -INFINITY;
    for (int w2 = 0; w2 < TW; ++w2) mm = fmaxf(mm, merge[(hl + w2 * HG) * stride_w + h]);
    float ll = 0.f;
    float acc[DL];
#pragma unroll
    for (int e = 0; e < DL; ++e) acc[e] = 0.f;
    for (int w2 = 0; w2 < TW; ++w2) {
      const float* mg = merge + (hl + w2 * HG) * stride_w;
      const float a = (mg[h] == -INFINITY) ? 0.f : ex2(mg[h] - mm);
      ll = fmaf(mg[G + h], a, ll);
      if (d0 < D) {
#pragma unroll
        for (int e = 0; e < DL; ++e) acc[e] = fmaf(mg[2 * G + h * D + d0 + e], a, acc[e]);
      }
    }
    const int hq = kvh * G + h;
    const float inv = ll > 0.f ? 1.f / ll : 0.f;
    float ov[DL];
#pragma unroll
    for (int e = 0; e < DL; ++e) ov[e] = acc[e] * inv;
    if (d0 < D) {
      if (p.num_splits == 1) {
        __nv_bfloat16* orow =
            static_cast<__nv_bfloat16*>(p.out) + ((int64_t)r * p.q_heads + hq) * D;
        Storage<__nv_bfloat16>::template store<DL>(orow + d0, ov);
      } else {
        const int64_t rs = ((int64_t)r * p.q_heads + hq) * p.num_splits + split;
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

}  // namespace npk
