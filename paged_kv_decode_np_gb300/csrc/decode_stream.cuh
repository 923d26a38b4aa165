// decode_stream.cuh -- the balanced streamed read (bf16 pools, head_dim a
// multiple of 64, kv heads in groups of 8): the same arithmetic as the split
// read (decode_mma.cuh), with the work laid out so that every SM gets the same
// number of history tokens and no thread block is launched for nothing.
//
// Partition (computed on the device from context_lens; no host sync, so the
// step stays graph-capturable).  Virtual rows v = hgi*rows + r (row r, kv
// head group hgi) are laid end to end, v's length being the row's context.
// With W their total and P = gridDim.x (one CTA per SM), CTA b owns the
// tokens from point(b*W/P) up to point((b+1)*W/P), where point(u) is the
// (virtual row, token) holding stream position u, the token rounded down to a
// whole chunk so that TMA boxes stay block-aligned.  A CTA walks its rows
// back to back with one producer/consumer pipeline: no drain between rows.
//
// Results.  A row that lies wholly inside one CTA is written straight to
// `out`.  Only the first and the last row of a CTA can be cut; for those the
// consumer warp of each kv head stores its unnormalised partial (running max
// m in log2 units, sum l, accumulator O) in the CTA's slot 0 (its first row)
// or slot 1 (its last row), and the CTA records its start point.  A second,
// small kernel then merges each cut row -- owned by the CTA where the row
// begins, one warp per kv head -- over the covering CTAs in CTA order
// (lse-weighted, the split read's combine), so results are deterministic
// and no thread block ever waits for another.
#pragma once

#include "decode_mma.cuh"

namespace npk {

constexpr int kStreamMaxVRows = 4096;  // virtual rows (row, 8-head group) per launch
constexpr int kStreamMaxCtas = 256;    // grid cap (the workspace is sized for it)

// The merge launch is a programmatic dependent of the read: it may be
// scheduled once every CTA of the read has started, and waits in
// griddepcontrol.wait until the read has finished and its writes are
// visible.  This hides the merge's launch latency behind the read's tail.
#ifndef NPK_STREAM_PDL
#define NPK_STREAM_PDL 1
#endif

// Workspace of the streamed read (host and device agree on this):
//   parts  [kStreamMaxCtas][2 slots][8 kv heads] entries of
//          m[16] l[16] o[16][D] fp32 (16 = mma rows)
//   pts    [kStreamMaxCtas + 1] longlong2: CTA b's start point (v, t)
// Nothing in it needs to start zeroed.
struct StreamWs {
  __host__ __device__ static constexpr size_t entry_floats(int d) {
    return (size_t)kMmaRows * 2 + (size_t)kMmaRows * d;
  }
  __host__ __device__ static constexpr size_t parts_bytes(int d) {
    return (size_t)kStreamMaxCtas * 2 * 8 * entry_floats(d) * sizeof(float);
  }
  __host__ __device__ static constexpr size_t bytes(int d) {
    return parts_bytes(d) + (size_t)(kStreamMaxCtas + 1) * 2 * sizeof(int64_t);
  }
};

__device__ __forceinline__ bool point_before(int64_t v1, int64_t t1, int64_t v2, int64_t t2) {
  return v1 < v2 || (v1 == v2 && t1 < t2);
}

template <int D, int G>
struct StreamSmem {
  using S = MmaSmem<D, G, true>;
  // ring (1024-aligned) | barriers | abort | virtual-row prefix (int64, V + 1)
  __host__ __device__ static constexpr size_t total(int stages, int vrows) {
    return S::total(8, stages, 8) + 16 + (size_t)(vrows + 1) * sizeof(int64_t);
  }
};

template <int D, int G, bool TWO>
__global__ void __launch_bounds__(kMaxThreads, 1)
    paged_decode_stream_kernel(const __grid_constant__ DecodeParams p) {
  using C = MmaCfg<D, G, true>;
  using S = MmaSmem<D, G, true>;
  constexpr unsigned FULL = 0xffffffffu;
  constexpr int HG = 8;

  const int b = blockIdx.x;
  const int P = gridDim.x;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int R = p.rows;
  const int NHG = p.kv_heads / HG;
  const int V = R * NHG;
  const int Q = p.query_len;
  const int MR = G * Q;
  const int64_t cap = (int64_t)p.max_blocks_per_row * p.block_size;
#if NPK_STREAM_PDL
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
#endif

  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const int stages = p.stages;
  const size_t stage_bytes = S::stage_bytes(HG);
  const size_t ring = S::ring_bytes(HG, stages, HG);
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + ring);
  uint64_t* empty_bar = full_bar + stages;
  volatile int* abort = reinterpret_cast<volatile int*>(empty_bar + stages);
  int64_t* pre = reinterpret_cast<int64_t*>(smem + ring + 16ull * stages + 16);
  __shared__ int64_t tsum[kMaxThreads];
  __shared__ int64_t range[4];  // vb, tb, ve, te

  auto row_len = [&](int v) -> int64_t {
    int64_t c = p.context_lens[v % R];
    return c < 0 ? 0 : (c > cap ? cap : c);
  };

  // ---- prefix of the virtual rows' lengths (two-level block scan)
  {
    const int nt = blockDim.x;
    const int per = (V + nt - 1) / nt;
    const int v0 = threadIdx.x * per, v1 = min(V, v0 + per);
    int64_t sum = 0;
    for (int v = v0; v < v1; ++v) sum += row_len(v);
    tsum[threadIdx.x] = sum;
    __syncthreads();
    if (threadIdx.x == 0) {
      int64_t run = 0;
      for (int t = 0; t < nt; ++t) {
        const int64_t x = tsum[t];
        tsum[t] = run;
        run += x;
      }
      pre[V] = run;
    }
    __syncthreads();
    int64_t run = tsum[threadIdx.x];
    for (int v = v0; v < v1; ++v) {
      pre[v] = run;
      run += row_len(v);
    }
    if (threadIdx.x == 0 && b == 0)  // out-of-range contexts were clamped
      for (int r = 0; r < R; ++r)
        if (p.context_lens[r] < 0 || p.context_lens[r] > cap) set_flag(p.err, NP_FLAG_CONTEXT);
  }
  __syncthreads();

  // ---- the partition: point(b) = (virtual row, chunk-aligned token) where
  // CTA b starts; CTA b owns [point(b), point(b+1))
  const int64_t total = pre[V];
  auto point = [&](int bb, int& pv, int64_t& pt) {
    const int64_t u = (int64_t)bb * total / P;  // total < 2^43, bb <= 256: no overflow
    int lo = 0, hi = V;  // the last v with pre[v] <= u
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (pre[mid] <= u) lo = mid;
      else hi = mid - 1;
    }
    pv = lo;
    pt = lo < V ? (u - pre[lo]) / C::CT * C::CT : 0;
  };
  if (threadIdx.x == 0) {
    int pv;
    int64_t pt;
    point(b, pv, pt);
    range[0] = pv;
    range[1] = pt;
    p.st_pts[2 * b] = pv;  // for the merge kernel
    p.st_pts[2 * b + 1] = pt;
    point(b + 1, pv, pt);
    range[2] = pv;
    range[3] = pt;
    if (b == P - 1) {
      p.st_pts[2 * P] = pv;
      p.st_pts[2 * P + 1] = pt;
    }
  }
  __syncthreads();
  const int vb = (int)range[0], ve = (int)range[2];
  const int64_t tb = range[1], te = range[3];

  // segment k of this CTA (rows vb..ve): token range [ts, tend) of row v
  auto seg_bounds = [&](int v, int64_t& ts, int64_t& tend) {
    ts = (v == vb) ? tb : 0;
    tend = (v == ve) ? te : row_len(v);
  };

  // ---- rows with no history: zeros (spread over the CTAs)
  for (int v = b; v < V; v += P) {
    if (row_len(v) != 0) continue;
    const int r = v % R, hgi = v / R;
    for (int qi = 0; qi < Q; ++qi) {
      __nv_bfloat16* o = static_cast<__nv_bfloat16*>(p.out) +
                         (((int64_t)r * Q + qi) * p.q_heads + hgi * HG * G) * D;
      for (int i = threadIdx.x; i < HG * G * D; i += blockDim.x) o[i] = __float2bfloat16_rn(0.f);
    }
  }

  // ---- fused append of the new tokens this CTA's segments hold
  for (int v = vb; v <= ve && v < V; ++v) {
    int64_t ts, tend;
    seg_bounds(v, ts, tend);
    if (ts < tend) fused_append<D, 2>(p, v % R, v / R, HG, row_len(v), ts, tend);
  }

  if (threadIdx.x == 0) {
    for (int i = 0; i < stages; ++i) {
      mbar_init(smem_u32(&full_bar[i]), 1);
      mbar_init(smem_u32(&empty_bar[i]), HG);  // one arrive per consumer warp
    }
    *abort = 0;
    fence_mbar_init();
  }
  __syncthreads();

  StageLayout<D, true> L;
  L.BT = p.box_tokens;
  L.half_bytes = (uint32_t)C::CT * HG * 128;
  L.box_bytes = (uint32_t)L.BT * HG * 128;
  L.RS = 0;
  L.hl = warp % HG;
  if (L.BT < 1 || L.BT > C::CT || C::CT % L.BT != 0) {
    if (threadIdx.x == 0) set_flag(p.err, NP_FLAG_CONFIG);
    return;
  }

  if (warp == HG) {
    // ======================= producer warp: every chunk of every segment
    const uint64_t pol = policy_evict_first();
    int64_t gch = 0, issued = 0;
    bool stop = false;
    for (int v = vb; v <= ve && v < V && !stop; ++v) {
      int64_t ts, tend;
      seg_bounds(v, ts, tend);
      const int r = v % R, hgi = v / R;
      const int64_t nblk = (row_len(v) + p.block_size - 1) / p.block_size;
      int64_t win = -1;
      int32_t my_id = 0;
      for (int64_t cb = ts; cb < tend; cb += C::CT, ++gch) {
        const int st = (int)(gch % stages);
        if (gch >= stages) {
          bool ok =
              mbar_wait(smem_u32(&empty_bar[st]), (uint32_t)((gch / stages - 1) & 1), abort);
          if (!__all_sync(FULL, ok)) {
            stop = true;
            break;
          }
        }
        const int n = (int)min((int64_t)C::CT, tend - cb);
        const uint32_t kdst = smem_u32(smem + st * stage_bytes);
        produce_chunk<D, true>(p, L, r, hgi, HG, cb, n, nblk, kdst,
                               kdst + (uint32_t)(stage_bytes / 2), smem_u32(&full_bar[st]), pol,
                               win, my_id, lane);
        issued = gch + 1;
      }
    }
    if (*abort) {  // never leave copies in flight (bounded)
      for (int64_t ch = max((int64_t)0, issued - stages); ch < issued; ++ch)
        mbar_wait_drain(smem_u32(&full_bar[ch % stages]), (uint32_t)((ch / stages) & 1));
    }
    return;
  }

  // ======================= consumer warp hl: its kv head of every segment
  const int hl = warp;
  const int g4 = lane >> 2, c4 = lane & 3;
  MmaWarp<D, G, TWO> W;
  int64_t gch = 0;
  bool first = true;
  for (int v = vb; v <= ve && v < V; ++v) {
    int64_t ts, tend;
    seg_bounds(v, ts, tend);
    if (ts >= tend) continue;
    const int r = v % R, hgi = v / R;
    const int kvh = hgi * HG + hl;
    const int64_t c = row_len(v);
    W.begin(p, r, kvh, c, lane);
    bool ok = true;
    for (int64_t cb = ts; cb < tend; cb += C::CT, ++gch) {
      const int st = (int)(gch % stages);
      ok = mbar_wait(smem_u32(&full_bar[st]), (uint32_t)((gch / stages) & 1), abort);
      if (!__all_sync(FULL, ok)) {
        set_flag(p.err, NP_FLAG_TIMEOUT);
        ok = false;
        break;
      }
      const int nvalid = (int)min((int64_t)C::CT, tend - cb);
      const uint32_t kst = smem_u32(smem + st * stage_bytes);
      for (int sb = 0; sb < nvalid; sb += C::ST)
        W.template tile<true>(L, kst, kst + (uint32_t)(stage_bytes / 2), sb, nvalid, cb,
                              p.qscale, lane);
      __syncwarp();  // every lane's reads of this stage are done
      if (lane == 0) mbar_arrive(smem_u32(&empty_bar[st]));
    }
    if (!ok) return;
    W.finish();

    if (ts == 0 && tend == c) {
      // ---- the whole row is here: normalise and store
      const float l_lo = __shfl_sync(FULL, W.lA, 8 * c4), l_hi = __shfl_sync(FULL, W.lA, 8 * c4 + 4);
      const float lb_lo = __shfl_sync(FULL, W.lB, 8 * c4), lb_hi = __shfl_sync(FULL, W.lB, 8 * c4 + 4);
      auto put = [&](int row, int d, float x, float l) {
        if (row >= MR) return;
        const int qi = row / G, h = row - qi * G;
        __nv_bfloat16* o = static_cast<__nv_bfloat16*>(p.out) +
                           (((int64_t)r * Q + qi) * p.q_heads + kvh * G + h) * D;
        o[d] = __float2bfloat16_rn(l > 0.f ? x / l : 0.f);
      };
#pragma unroll
      for (int mi = 0; mi < C::KS; ++mi) {
        const int d = 16 * mi + g4;
        put(2 * c4, d, W.oA[mi][0], l_lo);
        put(2 * c4 + 1, d, W.oA[mi][1], l_hi);
        put(2 * c4, d + 8, W.oA[mi][2], l_lo);
        put(2 * c4 + 1, d + 8, W.oA[mi][3], l_hi);
        if constexpr (TWO) {
          put(8 + 2 * c4, d, W.oB[mi][0], lb_lo);
          put(9 + 2 * c4, d, W.oB[mi][1], lb_hi);
          put(8 + 2 * c4, d + 8, W.oB[mi][2], lb_lo);
          put(9 + 2 * c4, d + 8, W.oB[mi][3], lb_hi);
        }
      }
      first = false;
      continue;
    }

    // ---- a cut row: store the partial for the merge kernel
    const int slot = first ? 0 : 1;
    first = false;
    const int64_t entry = ((int64_t)b * 2 + slot) * HG + hl;
    float* ent = p.ws_o + entry * (int64_t)StreamWs::entry_floats(D);
    W.store_rows(ent, ent + kMmaRows, ent + 2 * kMmaRows, MR, lane);
  }
}

// Merge of the cut rows.  Grid (the read's CTAs, G*Q mma rows); CTA b of
// the read is blockIdx.x here, and 8 warps = 8 kv heads.  CTA b owns the
// row its read range ends inside if that row also begins inside it
// (point(b) <= (v, 0) < point(b+1) < (v, c)); the row's partials are those
// of CTAs b, b+1, ... while they start before the row's end, each in slot 0
// when the row is that CTA's first and slot 1 otherwise.  Warp hl merges
// mma row blockIdx.y of its kv head: lanes take the covering CTAs for the
// max and the weights, then head_dim for the weighted sum of the partials,
// which runs over the CTAs in ascending order (a fixed order: results are
// deterministic).
template <int D, int G>
__global__ void __launch_bounds__(256) paged_decode_stream_merge_kernel(
    const __grid_constant__ DecodeParams p) {
  constexpr unsigned FULL = 0xffffffffu;
  constexpr int HG = 8;
  constexpr int DL = D / 32;
  constexpr int UNROLL = 8;
  const int b = blockIdx.x;
  const int row = blockIdx.y;
  const int P = gridDim.x;
  const int hl = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
#if NPK_STREAM_PDL
  asm volatile("griddepcontrol.wait;" ::: "memory");  // the read is complete
#endif
  const int64_t* pts = p.st_pts;
  const int64_t vb = pts[2 * b], tb = pts[2 * b + 1];
  const int64_t v = pts[2 * b + 2], te = pts[2 * b + 3];
  const int R = p.rows;
  if (te == 0 || v >= (int64_t)R * (p.kv_heads / HG)) return;  // b's range ends at a row boundary
  if (!point_before(vb, tb, v, 0) && !(vb == v && tb == 0)) return;  // v began before b
  const int64_t cap = (int64_t)p.max_blocks_per_row * p.block_size;
  int64_t c = p.context_lens[v % R];
  c = c < 0 ? 0 : (c > cap ? cap : c);
  const int r = (int)(v % R), hgi = (int)(v / R);
  const int kvh = hgi * HG + hl;
  const int Q = p.query_len;
  if (row >= G * Q) return;
  const int64_t ent_floats = (int64_t)StreamWs::entry_floats(D);

  // the covering CTAs b..bl: those that start before (v, c)
  int bl = b;
  for (int base = b + 1; base < P; base += 32) {
    const int j = base + lane;
    const bool cov = j < P && point_before(pts[2 * j], pts[2 * j + 1], v, c);
    const unsigned m = __ballot_sync(FULL, cov);
    const int n = __ffs(~m) - 1;  // leading covering lanes (-1: all 32)
    if (n < 0) {
      bl = base + 31;
      continue;
    }
    bl = base + n - 1;
    break;
  }
  // lane j's partial of CTA base + j: entry offset (-1 for none), m and l
  auto load_ml = [&](int base, int64_t& off, float& mj, float& lj) {
    const int j = base + lane;
    off = -1;
    mj = -INFINITY;
    lj = 0.f;
    if (j > bl) return;
    const int64_t v0 = pts[2 * j], t0 = pts[2 * j + 1];
    if (!point_before(v0, t0, pts[2 * j + 2], pts[2 * j + 3])) return;  // an empty range
    const int sl = (v0 == v) ? 0 : 1;
    off = (((int64_t)j * 2 + sl) * HG + hl) * ent_floats;
    mj = p.ws_o[off + row];
    lj = p.ws_o[off + kMmaRows + row];
  };
  float mm = -INFINITY;
  for (int base = b; base <= bl; base += 32) {
    int64_t off;
    float mj, lj;
    load_ml(base, off, mj, lj);
    mm = fmaxf(mm, mj);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mm = fmaxf(mm, __shfl_xor_sync(FULL, mm, o));

  const int d0 = lane * DL;
  float lsum = 0.f, acc[DL];
#pragma unroll
  for (int e2 = 0; e2 < DL; ++e2) acc[e2] = 0.f;
  for (int base = b; base <= bl; base += 32) {
    int64_t off;
    float mj, lj;
    load_ml(base, off, mj, lj);
    const float aj = (off < 0 || mj == -INFINITY) ? 0.f : ex2(mj - mm);
    lsum = fmaf(aj, lj, lsum);
    const int n = min(32, bl - base + 1);
    for (int k = 0; k < n; k += UNROLL) {
      float ak[UNROLL], ok[UNROLL][DL];
#pragma unroll
      for (int u = 0; u < UNROLL; ++u) {  // the loads of UNROLL partials first
        const int src = (k + u) & 31;
        ak[u] = __shfl_sync(FULL, aj, src);
        const int64_t of = __shfl_sync(FULL, off, src);
        const bool use = k + u < n && ak[u] != 0.f;
        const float* e = p.ws_o + (use ? of : 0) + 2 * kMmaRows + row * D + d0;
#pragma unroll
        for (int e2 = 0; e2 < DL; ++e2) ok[u][e2] = use ? e[e2] : 0.f;
        if (!use) ak[u] = 0.f;
      }
#pragma unroll
      for (int u = 0; u < UNROLL; ++u)  // then their sum, in CTA order
#pragma unroll
        for (int e2 = 0; e2 < DL; ++e2) acc[e2] = fmaf(ok[u][e2], ak[u], acc[e2]);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) lsum += __shfl_xor_sync(FULL, lsum, o);
  const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
  float ov[DL];
#pragma unroll
  for (int e2 = 0; e2 < DL; ++e2) ov[e2] = acc[e2] * inv;
  const int qi = row / G, h = row - qi * G;
  __nv_bfloat16* o = static_cast<__nv_bfloat16*>(p.out) +
                     (((int64_t)r * Q + qi) * p.q_heads + kvh * G + h) * D;
  Storage<__nv_bfloat16>::template store<DL>(o + d0, ov);
}

}  // namespace npk
