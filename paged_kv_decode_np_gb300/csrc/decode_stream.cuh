// decode_stream.cuh -- the balanced streamed read (kv heads in groups of HG,
// the largest divisor of the count up to 8; bf16 pools with head_dim a
// multiple of 64 on the tensor cores, through tiled TMA boxes, or fp32 pools
// with head_dim a multiple of 32 on the FMA pipes, through 1-D bulk
// copies): the same arithmetic as the split read,
// with the work laid out so that every SM gets the same number of history
// tokens and no thread block is launched for nothing.
//
// Partition (computed on the device from context_lens; no host sync, so the
// step stays graph-capturable).  Virtual rows v = hgi*rows + r (row r, kv
// head group hgi) are laid end to end, each as ceil(context / CT) chunks of
// CT tokens (a stage: its last chunk may be short).  With W chunks in all
// and P = gridDim.x (one CTA per SM), the first Pe = min(P, ceil(W /
// kMinCtaChunks)) CTAs share the stream -- a small step gives each working
// CTA a few chunks instead of spreading a short row over every SM -- and CTA
// b < Pe owns chunks [floor(b*W/Pe), floor((b+1)*W/Pe)); chunk starts are
// whole chunks of their row, so TMA boxes stay block-aligned; CTAs b >= Pe
// own nothing.  A CTA walks its rows back to back with one producer/consumer
// pipeline: no drain between rows.
//
// Results.  A row that lies wholly inside one CTA is written straight to
// `out`.  Only the first and the last row of a CTA can be cut; for those the
// consumer warps of each kv head store its unnormalised partial (running max
// m in log2 units, sum l, accumulator O; merged first across the head's
// warps when several read it) in the CTA's slot 0 (its first row) or slot 1
// (its last row), and the CTA that owns a cut row (the one where the row
// begins) leaves a descriptor of it.  A second, small kernel then
// merges each cut row -- in tasks of a few mma rows of one kv head, dealt
// over all its blocks -- over the covering CTAs in CTA order (the split
// read's max-and-weights combine), so results are deterministic and no
// thread block ever waits for another.
#pragma once

#include "decode_fma.cuh"
#include "decode_mma.cuh"

namespace npk {

constexpr int kStreamMaxVRows = 4096;  // virtual rows (row, kv-head group) per launch
constexpr int kStreamMaxCtas = 160;    // grid cap, >= the GB300's 152 SMs (the
                                       // workspace is sized for it)

// The merge launch is a programmatic dependent of the read: it may be
// scheduled once every CTA of the read has started, and waits in
// griddepcontrol.wait until the read has finished and its writes are
// visible.  This hides the merge's launch latency behind the read's tail.
#ifndef NPK_STREAM_PDL
#define NPK_STREAM_PDL 1
#endif

// Merge tasks may cover half the head_dim (rows cut into many pieces).
#ifndef NPK_MERGE_DH2
#define NPK_MERGE_DH2 1
#endif

// Cut-row partials and merge descriptors are stored with an L2 evict-last
// hint (the merge reads them back after the read has streamed the pools).
#ifndef NPK_PARTIAL_KEEP
#define NPK_PARTIAL_KEEP 1
#endif
#if NPK_PARTIAL_KEEP
using PartialStore = L2KeepStore;
#else
struct PartialStore : PlainStore {
  __device__ __forceinline__ static PartialStore make() { return PartialStore(); }
  __device__ __forceinline__ void i4(int4* p, int4 v) const { *p = v; }
};
#endif

// Merge blocks have 256 * NPK_MERGE_RPB threads (16 warps by default),
// which share the block's merge tasks.
#ifndef NPK_MERGE_RPB
#define NPK_MERGE_RPB 2
#endif
constexpr int kMergeRpb = NPK_MERGE_RPB;

// Workspace of the streamed read (host and device agree on this):
//   parts  [kStreamMaxCtas][2 slots][8 kv heads] entries of
//          m[16] l[16] o[16][D] fp32 (16 = mma rows)
//   desc   [kStreamMaxCtas] int4: CTA b's merge descriptor {v, b, bl, slot}
//          for the cut row it owns (v = -1: none)
// Nothing in it needs to start zeroed.
struct StreamWs {
  __host__ __device__ static constexpr size_t entry_floats(int d) {
    return (size_t)kMmaRows * 2 + (size_t)kMmaRows * d;
  }
  __host__ __device__ static constexpr size_t parts_bytes(int d) {
    return (size_t)kStreamMaxCtas * 2 * 8 * entry_floats(d) * sizeof(float);
  }
  __host__ __device__ static constexpr size_t bytes(int d) {  // + one int4 descriptor per CTA
    return parts_bytes(d) + (size_t)kStreamMaxCtas * 4 * sizeof(int32_t);
  }
};


// Per storage type: tokens per stage, the stage size and the consumer warp.
template <typename T, int D, int G, bool TWO>
struct StreamKind;

template <int D, int G, bool TWO>
struct StreamKind<__nv_bfloat16, D, G, TWO> {  // tensor cores, tiled TMA boxes
  static constexpr bool kTmap = true;
  using Warp = MmaWarp<D, G, TWO>;
  static constexpr int CT = MmaCfg<D, G, true>::CT;
  static constexpr int ST = MmaCfg<D, G, true>::ST;
  __host__ __device__ static constexpr size_t stage_bytes(int hg) {
    return MmaSmem<D, G, true>::stage_bytes(hg);
  }
  __host__ __device__ static constexpr size_t tile_floats() { return 0; }
};

template <int D, int G, bool MQ>
struct StreamKind<float, D, G, MQ> {  // FMA pipes, 1-D bulk copies of token rows
  // MQ: several query tokens per row, (query token, head) rows up to 8
  static constexpr bool kTmap = false;
  using Warp = FmaWarp<D, G, MQ>;
  static constexpr int CT = FmaCfg<D, G, MQ>::CT;
  static constexpr int ST = CT;
  __host__ __device__ static constexpr size_t stage_bytes(int hg) {
    return 2ull * CT * hg * D * sizeof(float);
  }
  __host__ __device__ static constexpr size_t tile_floats() { return FmaCfg<D, G, MQ>::TILE; }
};

// A consumer warp's row-end state in shared memory: m[MRP] (log2 units),
// l[MRP], O[MR][D] floats, MRP = MR rounded up to 4 so that every part and
// every entry starts on a 16-byte boundary (the fp32 warp stores O rows as
// 16-byte vectors; D is a multiple of 32).
__host__ __device__ constexpr int wstate_mrp(int mr) { return (mr + 3) & ~3; }
__host__ __device__ constexpr size_t wstate_entry_floats(int mr, int d) {
  return 2 * (size_t)wstate_mrp(mr) + (size_t)mr * d;
}

// Shared memory: ring (1024-aligned) | full, empty barriers | abort |
// virtual rows' chunk prefix (int64, V + 1) | their lengths (int32, V) |
// consumer tiles (16-aligned) | the token warps' states (tw > 1).  hg = kv
// heads per CTA, tw = consumer warps per kv head times the pieces of K::CT
// tokens each of them takes per stage: a stage holds tw * K::CT tokens.
template <typename T, int D, int G, bool TWO>
struct StreamSmem {
  using K = StreamKind<T, D, G, TWO>;
  // sm: K::CT-token pieces per kv head in a stage (consumer warps per head
  // times the pieces each takes)
  __host__ __device__ static constexpr size_t stage_bytes(int hg, int sm) {
    return K::stage_bytes(hg) * sm;
  }
  __host__ __device__ static constexpr size_t lens_offset(int hg, int sm, int stages, int vrows) {
    return stage_bytes(hg, sm) * stages + 16ull * stages + 16 + (size_t)(vrows + 1) * 8;
  }
  __host__ __device__ static constexpr size_t tiles_offset(int hg, int sm, int stages, int vrows) {
    return (lens_offset(hg, sm, stages, vrows) + (size_t)vrows * 4 + 15) / 16 * 16;
  }
  // several consumer warps per kv head (tw > 1): their (m, l, O) rows at a
  // row boundary, one entry per warp
  __host__ __device__ static constexpr size_t merge_offset(int hg, int sm, int stages, int vrows) {
    return (tiles_offset(hg, sm, stages, vrows) + 8 * K::tile_floats() * sizeof(float) + 15) /
           16 * 16;
  }
  // tw > 1: ncw consumer warps' row-end states of mr rows each
  __host__ __device__ static constexpr size_t total(int hg, int sm, int stages, int vrows,
                                                    int tw, int ncw, int mr) {
    return 1024 + merge_offset(hg, sm, stages, vrows) +
           (tw > 1 ? (size_t)ncw * wstate_entry_floats(mr, D) * sizeof(float) : 0) +
           (tw > 1 ? 16 : 0);  // + the merge's two mbarriers
  }
};

// The TW consumer warps of kv head hl (warps hl, hl + HG, ...) left their
// unnormalised states side by side in `ws`, one entry per warp (the layout
// of wstate_entry_floats); warp tw merges
// rows tw, tw + TW, ... of them in warp order (max and weights) and stores
// each row: normalised to `out` when the whole row is this CTA's, else
// unnormalised to the cut row's partial entry `ent` (the workspace layout:
// m[16], l[16], O[16][D]) for the merge kernel.
template <typename T, int D, typename St>
__device__ __forceinline__ void merge_warp_states(const DecodeParams& p, const float* ws, int hl,
                                                  int HG, int TW, int tw, int MR, int Gr,
                                                  int64_t r, int kvh, bool whole, float* ent,
                                                  St keep, int lane) {
  constexpr int RW = kMmaRows;
  constexpr int DL = D >= 32 ? D / 32 : 1;  // dims per lane
  const int64_t stride = (int64_t)wstate_entry_floats(MR, D);
  const int MRP = wstate_mrp(MR);
  const int Q = p.query_len;
  const int d0 = lane * DL;
  for (int row = tw; row < MR; row += TW) {
    float mm = -INFINITY;
    for (int w2 = 0; w2 < TW; ++w2) mm = fmaxf(mm, ws[(hl + w2 * HG) * stride + row]);
    const float msub = mm == -INFINITY ? 0.f : mm;
    float ll = 0.f, acc[DL];
#pragma unroll
    for (int e = 0; e < DL; ++e) acc[e] = 0.f;
    for (int w2 = 0; w2 < TW; ++w2) {
      const float* w = ws + (hl + w2 * HG) * stride;
      const float a = ex2(w[row] - msub);  // a state with nothing in it: m = -inf, a = 0
      ll = fmaf(w[MRP + row], a, ll);
      if (d0 < D) {
#pragma unroll
        for (int e = 0; e < DL; ++e) acc[e] = fmaf(w[2 * MRP + row * D + d0 + e], a, acc[e]);
      }
    }
    if (whole) {
      const float inv = ll > 0.f ? 1.f / ll : 0.f;
      float ov[DL];
#pragma unroll
      for (int e = 0; e < DL; ++e) ov[e] = acc[e] * inv;
      const int qi = row / Gr, h = row - qi * Gr;
      T* o = static_cast<T*>(p.out) + ((r * Q + qi) * p.q_heads + (int64_t)kvh * Gr + h) * D;
      if (d0 < D) Storage<T>::template store<DL>(o + d0, ov);
    } else {
      if (lane == 0) {
        keep(&ent[row], mm);
        keep(&ent[RW + row], ll);
      }
      if (d0 < D) {
#pragma unroll
        for (int e = 0; e < DL; ++e) keep(&ent[2 * RW + row * D + d0 + e], acc[e]);
      }
    }
  }
}

// MULTI: built for several consumer warps per kv head (p.token_warps > 1,
// row-end merges of their states); without it the kernel holds none of
// that code and reads one warp per head.
template <typename T, int D, int G, bool TWO, bool MULTI>
__global__ void __launch_bounds__(kMaxThreads, 1)
    paged_decode_stream_kernel(const __grid_constant__ DecodeParams p) {
  using K = StreamKind<T, D, G, TWO>;
  using C = K;  // chunk geometry (CT, ST)
  constexpr unsigned FULL = 0xffffffffu;
  const int HG = p.head_group;   // kv heads per CTA (the largest divisor of kv_heads <= 8)
  const int TW = MULTI ? p.token_warps : 1;  // consumer warps per kv head (HG * TW <= 8)
  const int NCW = HG * TW;       // consumer warps 0 .. NCW-1: warp w reads kv head w % HG
  constexpr int kProducer = kMaxConsumerWarps;  // warp 8

  const int b = blockIdx.x;
  const int P = gridDim.x;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int R = p.rows;
  const int NHG = p.kv_heads / HG;
  const int V = R * NHG;
  const int Q = p.query_len;
  const int Gr = G > 0 ? G : p.q_heads / p.kv_heads;  // G = 0: the group set at run time
  const int MR = Gr * Q;
  const int64_t cap = (int64_t)p.max_blocks_per_row * p.block_size;
#if NPK_STREAM_PDL
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
#endif

  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const int stages = p.stages;
  // a stage: WS = SL * K::CT tokens for each of a head's TW consumer warps
  const int WS = C::CT * p.stage_slices;
  const int CT = WS * TW;
  using SS = StreamSmem<T, D, G, TWO>;
  const int SM = TW * p.stage_slices;  // K::CT-token pieces per kv head in a stage
  const size_t stage_bytes = SS::stage_bytes(HG, SM);
  const size_t ring = stage_bytes * stages;
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + ring);
  uint64_t* empty_bar = full_bar + stages;
  volatile int* abort = reinterpret_cast<volatile int*>(empty_bar + stages);
  int64_t* pre = reinterpret_cast<int64_t*>(smem + ring + 16ull * stages + 16);
  int32_t* lens = reinterpret_cast<int32_t*>(smem + SS::lens_offset(HG, SM, stages, V));
  float* tiles = reinterpret_cast<float*>(smem + SS::tiles_offset(HG, SM, stages, V));
  float* wstate =  // TW > 1: the consumer warps' states at a row boundary
      reinterpret_cast<float*>(smem + SS::merge_offset(HG, SM, stages, V));
  // (one 16-byte aligned entry per consumer warp)
  uint64_t* seg_bar = reinterpret_cast<uint64_t*>(wstate + (size_t)NCW * wstate_entry_floats(MR, D));
  __shared__ int64_t wsum[32];
  __shared__ int64_t range[4];  // vb, tb, ve, te

  auto row_len = [&](int v) -> int64_t {
    int64_t c = p.context_lens[v % R];
    return c < 0 ? 0 : (c > cap ? cap : c);
  };

  if (threadIdx.x == 0) {  // the ring's barriers (ordered by the scan's barriers)
    for (int i = 0; i < stages; ++i) {
      mbar_init(smem_u32(&full_bar[i]), 1);
      mbar_init(smem_u32(&empty_bar[i]), NCW);  // one arrive per consumer warp
    }
    if (TW > 1) {  // row boundaries: states written, then merged (all consumer warps)
      mbar_init(smem_u32(&seg_bar[0]), NCW);
      mbar_init(smem_u32(&seg_bar[1]), NCW);
    }
    *abort = 0;
    fence_mbar_init();
  }

  // ---- prefix of the virtual rows' chunk counts (ceil(length / CT)):
  // each thread sums a run of rows, warps scan the run sums with shuffles,
  // warp 0 scans the warp sums; the lengths stay in shared memory
  {
    const int nt = blockDim.x;
    const int per = (V + nt - 1) / nt;
    const int v0 = threadIdx.x * per, v1 = min(V, v0 + per);
    int64_t sum = 0;
    for (int v = v0; v < v1; ++v) {
      const int64_t len = row_len(v);
      lens[v] = (int32_t)len;
      sum += (len + CT - 1) / CT;
      if (b == 0 && v < R && (p.context_lens[v] < 0 || p.context_lens[v] > cap))
        set_flag(p.err, NP_FLAG_CONTEXT);  // clamped above
    }
    int64_t x = sum;  // inclusive scan within the warp
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int64_t y = __shfl_up_sync(FULL, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) wsum[warp] = x;
    __syncthreads();
    if (warp == 0) {
      const int nw = nt / 32;
      int64_t t = lane < nw ? wsum[lane] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int64_t y = __shfl_up_sync(FULL, t, o);
        if (lane >= o) t += y;
      }
      if (lane < nw) wsum[lane] = t;
      if (lane == nw - 1) pre[V] = t;
    }
    __syncthreads();
    int64_t run = x - sum + (warp > 0 ? wsum[warp - 1] : 0);
    for (int v = v0; v < v1; ++v) {
      pre[v] = run;
      run += ((int64_t)lens[v] + CT - 1) / CT;
    }
  }
  __syncthreads();

  // ---- the partition, in chunks (CT tokens; a row's last chunk may be
  // short): the rows' chunks laid end to end, CTA b takes chunks
  // [floor(b*W/Pe), floor((b+1)*W/Pe)) of the W in all -- equal chunk
  // counts to within one.  point(b) = (virtual row, first token) where CTA b
  // starts; CTA b owns [point(b), point(b+1))
  const int64_t total = pre[V];  // W
  constexpr int64_t kMinCtaChunks = 4;  // at least 4 chunks per working CTA
  const int Pe = (int)min((int64_t)P, max((int64_t)1, (total + kMinCtaChunks - 1) / kMinCtaChunks));
  auto point = [&](int bb, int& pv, int64_t& pt) {
    const int64_t u = bb >= Pe ? total : (int64_t)bb * total / Pe;  // total < 2^41: no overflow
    int lo = 0, hi = V;  // the last v with pre[v] <= u
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (pre[mid] <= u) lo = mid;
      else hi = mid - 1;
    }
    pv = lo;
    pt = lo < V ? (u - pre[lo]) * CT : 0;
  };
  if (threadIdx.x == 0 || threadIdx.x == 32) {  // the two ends, found in parallel
    const int k = threadIdx.x >> 5;
    int pv;
    int64_t pt;
    point(b + k, pv, pt);
    range[2 * k] = pv;
    range[2 * k + 1] = pt;
  }
  __syncthreads();
  const int vb = (int)range[0], ve = (int)range[2];
  const int64_t tb = range[1], te = range[3];
  // from here on a row's (clamped) length comes from shared memory, not
  // from another global load
  auto len_of = [&](int v) -> int64_t { return lens[v]; };

  // segment k of this CTA (rows vb..ve): token range [ts, tend) of row v
  auto seg_bounds = [&](int v, int64_t& ts, int64_t& tend) {
    ts = (v == vb) ? tb : 0;
    tend = (v == ve) ? te : len_of(v);
  };

  StageLayout<D, true> L;
  L.BT = p.box_tokens;
  L.slab_bytes = (uint32_t)L.BT * HG * 128;
  L.box_bytes = (uint32_t)(D / 64) * L.slab_bytes;
  L.RS = 0;
  L.hl = warp % HG;
  if (K::kTmap && (L.BT < 1 || L.BT > C::CT || C::CT % L.BT != 0)) {  // boxes tile a slice
    if (threadIdx.x == 0) {  // no partials: the merge finds no cut rows
      set_flag(p.err, NP_FLAG_CONFIG);
      reinterpret_cast<int4*>(p.st_desc)[b] = make_int4(-1, 0, 0, 0);
    }
    return;
  }

  // Warps 0..7 write the zero rows and the fused append (new tokens side by
  // side, one per group of warps) while the producer starts on the history;
  // they signal
  // named barrier 1 (after fence.proxy.async, so the appended rows are
  // visible to TMA) and the producer waits on it before the first chunk that
  // holds a new token.  Warps NCW..7 (HG * TW < 8) have no kv head and leave
  // after that.
  constexpr int kAppendBar = 1;
  if (warp < kProducer) {
    const int tid = threadIdx.x, nthr = 32 * kProducer;
    for (int v = b; v < V; v += P) {  // rows with no history: zeros
      if (len_of(v) != 0) continue;
      const int r = v % R, hgi = v / R;
      for (int qi = 0; qi < Q; ++qi) {
        T* o = static_cast<T*>(p.out) + (((int64_t)r * Q + qi) * p.q_heads + hgi * HG * Gr) * D;
        for (int i = tid; i < HG * Gr * D; i += nthr) o[i] = T(0.f);
      }
    }
    if (p.slot_mapping != nullptr) {
      // the new tokens whose positions lie in this CTA's segments, one per
      // group of GW warps in turn (token k of the walk goes to group k % NG;
      // GW: enough warps that no thread copies more than kAppendVpl vectors)
      const int nvec = HG * D * (int)sizeof(T) / 16;
      const int GW = nvec <= 32 * kAppendVpl ? 1 : nvec <= 64 * kAppendVpl ? 2
                   : nvec <= 128 * kAppendVpl ? 4 : 8;
      const int NG = kProducer / GW;
      const int grp = warp / GW, t = (warp % GW) * 32 + lane;
      bool wrote = false;
      int k = 0;
      for (int v = vb; v <= ve && v < V; ++v) {
        int64_t ts, tend;
        seg_bounds(v, ts, tend);
        const int64_t c = len_of(v);
        for (int j = 0; j < Q; ++j) {
          const int64_t pos = c - Q + j;
          if (pos < 0 || pos < ts || pos >= tend) continue;
          if (k++ % NG == grp)
            wrote |= append_token_group<D, (int)sizeof(T)>(p, v % R, v / R, HG, pos, j, t,
                                                           32 * GW);
        }
      }
      if (wrote) asm volatile("fence.proxy.async.global;" ::: "memory");
    }
    asm volatile("bar.arrive %0, %1;" ::"r"(kAppendBar), "r"(blockDim.x) : "memory");
    if (threadIdx.x == 0) {
      // Merge descriptor {v, b, bl, slot} of the row this CTA's range ends
      // inside, if it began here ((vb, tb) <= (v, 0)) and so cuts it: its
      // covering CTAs are b through bl, the last CTA whose stream position
      // floor(bb*W/Pe) lies before the row's end pre[v+1]; CTAs after b hold
      // v as their first row (slot 0), b holds it in slot 0 if it is b's
      // first row, else in slot 1.  v = -1: no such row.  Written here,
      // after the partition, so the 64-bit division stays off the
      // producer's start; the merge reads it only once the read has
      // finished.
      int4 d = make_int4(-1, 0, 0, 0);
      if (te > 0 && ve < V && (vb < ve || tb == 0)) {
        const int64_t x = pre[ve + 1];
        d.x = ve;
        d.y = b;
        d.z = (int)min((int64_t)Pe - 1, (x * Pe - 1) / total);
        d.w = vb == ve ? 0 : 1;
      }
      const PartialStore keep = PartialStore::make();  // read back by the merge
      keep.i4(reinterpret_cast<int4*>(p.st_desc) + b, d);
    }
    if (warp >= NCW) return;
  }

  if (warp == kProducer) {
    // ======================= producer warp: every chunk of every segment
    // Block-table entries come in windows of 32 blocks of one row, aligned
    // to multiples of 32 blocks; a chunk never straddles two (chunk starts
    // and 32-block spans are both multiples of CT tokens).  Lane j holds
    // entry j of the current window (cur) and of the window after it (nxt:
    // the row's next window, or the next segment's first), loaded one window
    // ahead so that issuing never waits on the table.  Positions fit int32
    // (the host admits tables of at most INT32_MAX tokens).
    const uint64_t pol = policy_evict_first();
    const int32_t bs = p.block_size;
    auto next_seg = [&](int v, int64_t& ts, int64_t& tend) -> int {  // first non-empty >= v
      for (; v <= ve && v < V; ++v) {
        seg_bounds(v, ts, tend);
        if (ts < tend) return v;
      }
      ts = tend = 0;
      return -1;
    };
    auto load_window = [&](int v, int32_t w) -> int32_t {
      if (v < 0) return 0;
      const int32_t j = w + lane;
      return j < (int32_t)((len_of(v) + bs - 1) / bs)
                 ? p.block_tables[(int64_t)(v % R) * p.max_blocks_per_row + j]
                 : 0;
    };
    int64_t ts64, te64;
    int v = next_seg(vb, ts64, te64);
    int32_t ts = (int32_t)ts64, tend = (int32_t)te64;
    int32_t ww = v >= 0 ? ts / bs / 32 * 32 : 0;  // current window: row v, first block ww
    int32_t cur = load_window(v, ww), nxt = 0;
    int nv = -1;  // the window after it: row nv, first block nw
    int32_t nw = 0;
    int64_t gch = 0;
    int st = 0;
    uint32_t ph = 1;  // parity of stage st's empty barrier: (gch / stages - 1) & 1
    bool stop = false;
    const bool fused = p.slot_mapping != nullptr;
    bool appended = false;  // past named barrier 1 (exactly once)
    while (v >= 0 && !stop) {
      const int hgi = v / R;
      const int32_t lastw = (tend - 1) / bs / 32 * 32;
      const int32_t first_new = (int32_t)len_of(v) - Q;  // the row's first new position
      int64_t nts, nte;
      const int vn = next_seg(v + 1, nts, nte);
      auto set_next = [&]() {  // the window after (v, ww), loaded now
        if (ww < lastw) {
          nv = v;
          nw = ww + 32;
        } else {
          nv = vn;
          nw = vn >= 0 ? (int32_t)nts / bs / 32 * 32 : 0;
        }
        nxt = load_window(nv, nw);
      };
      set_next();
      for (int32_t cb = ts; cb < tend; cb += CT, ++gch) {
        if (gch >= stages) {
          bool ok = mbar_wait(smem_u32(&empty_bar[st]), ph, abort);
          if (!__all_sync(FULL, ok)) {
            stop = true;
            break;
          }
        }
        const int32_t w = cb / bs / 32 * 32;
        if (w != ww) {  // into the row's next window
          ww = w;
          cur = (nv == v && nw == w) ? nxt : load_window(v, w);
          set_next();
        }
        const int n = min(CT, tend - cb);
        if (fused && !appended && cb + n > first_new) {
          asm volatile("bar.sync %0, %1;" ::"r"(kAppendBar), "r"(blockDim.x) : "memory");
          appended = true;
        }
        const uint32_t kdst = smem_u32(smem + st * stage_bytes);
        const uint32_t vdst = kdst + (uint32_t)(stage_bytes / 2);
        const uint32_t fb = smem_u32(&full_bar[st]);
        if constexpr (K::kTmap) {
          const int nbox = (n + L.BT - 1) / L.BT;
          if (lane == 0) mbar_arrive_expect_tx(fb, 2u * nbox * L.box_bytes);
          const int items = nbox * 2;  // (box, K|V)
          for (int it0 = 0; it0 < items; it0 += 32) {
            const int it = it0 + lane;
            const int bx = (it < items ? it : 0) >> 1;
            const int32_t t = cb + bx * L.BT;
            const int32_t j = t / bs;
            int32_t blk = __shfl_sync(FULL, cur, j - ww);
            if (it < items) {
              if (blk < 0 || blk >= p.num_blocks) {
                set_flag(p.err, NP_FLAG_BLOCK_ID);
                blk = 0;
              }
              const bool isv = (it & 1) != 0;
              const int32_t slot = blk * bs + (t - j * bs);
              tma_load_4d((isv ? vdst : kdst) + bx * L.box_bytes, isv ? &p.tm_v : &p.tm_k, 0, slot,
                          hgi * HG, 0, fb, pol);
            }
          }
        } else {
          // stage rows [token][HG kv heads][D]: when the pool has just HG kv
          // heads a run of tokens inside one block is one contiguous copy
          // (lane k: the chunk's k-th block); else one copy per token (lane =
          // token, 32 tokens a round).  A chunk lies in window ww.
          const uint32_t row_b = (uint32_t)HG * D * (uint32_t)sizeof(T);
          const int64_t pool_row = (int64_t)p.kv_heads * D * (int64_t)sizeof(T);
          const char* kp = static_cast<const char*>(p.k_pool) + (int64_t)hgi * row_b;
          const char* vp = static_cast<const char*>(p.v_pool) + (int64_t)hgi * row_b;
          if (lane == 0) mbar_arrive_expect_tx(fb, 2u * (uint32_t)n * row_b);
          const int32_t jf = cb / bs;
          const bool whole = p.kv_heads == HG;
          for (int g0 = 0; g0 < (whole ? 1 : n); g0 += 32) {
            const int32_t j = whole ? jf + lane : (cb + min(g0 + lane, n - 1)) / bs;
            int32_t blk = __shfl_sync(FULL, cur, (j - ww) & 31);
            int64_t ta, tz;  // this lane's tokens [ta, tz)
            if (whole) {
              ta = max((int64_t)cb, (int64_t)j * bs);
              tz = min((int64_t)cb + n, ((int64_t)j + 1) * bs);
            } else {
              ta = cb + g0 + lane;
              tz = g0 + lane < n ? ta + 1 : ta;
            }
            if (ta < tz) {
              if (blk < 0 || blk >= p.num_blocks) {
                set_flag(p.err, NP_FLAG_BLOCK_ID);
                blk = 0;
              }
              const int64_t slot = (int64_t)blk * bs + (ta - j * bs);
              const uint32_t off = (uint32_t)(ta - cb) * row_b;
              const uint32_t bytes = (uint32_t)(tz - ta) * row_b;
              bulk_g2s(kdst + off, kp + slot * pool_row, bytes, fb, pol);
              bulk_g2s(vdst + off, vp + slot * pool_row, bytes, fb, pol);
            }
          }
        }
        if (++st == stages) {
          st = 0;
          ph ^= 1u;
        }
      }
      // into the next segment: its first window was loaded as nxt
      v = vn;
      ts = (int32_t)nts;
      tend = (int32_t)nte;
      if (v >= 0) {
        const int32_t w = ts / bs / 32 * 32;
        cur = (nv == v && nw == w) ? nxt : load_window(v, w);
        ww = w;
      }
    }
    if (!appended)  // complete the barrier the consumers signalled
      asm volatile("bar.sync %0, %1;" ::"r"(kAppendBar), "r"(blockDim.x) : "memory");
    const int64_t issued = gch;
    if (*abort) {  // never leave copies in flight (bounded)
      for (int64_t ch = max((int64_t)0, issued - stages); ch < issued; ++ch)
        mbar_wait_drain(smem_u32(&full_bar[ch % stages]), (uint32_t)((ch / stages) & 1));
    }
    return;
  }

  // ======================= consumer warp (hl, tw): kv head hl of every
  // segment; warp tw takes tokens [tw*WS, (tw+1)*WS) of every stage (WS =
  // SL pieces of K::CT tokens), and with TW > 1 warps per head the head's
  // warps merge their states at the end of every segment
  const int hl = warp % HG, tw = warp / HG;
  const PartialStore keep = PartialStore::make();  // cut-row partials: read by the merge
  if (vb == ve && tb == te && vb < V && tw == 0) {
    // an empty range inside row vb: an empty partial (m = -inf, l = 0, o = 0)
    // in slot 0 for the merge of that row
    float* ent = p.ws_o + ((int64_t)b * 2 * HG + hl) * (int64_t)StreamWs::entry_floats(D);
    if (lane < kMmaRows) {
      keep(&ent[lane], -INFINITY);
      keep(&ent[kMmaRows + lane], 0.f);
    }
    for (int i = lane; i < kMmaRows * D; i += 32) keep(&ent[2 * kMmaRows + i], 0.f);
  }
  typename K::Warp W;
  float* tile = tiles + (size_t)warp * K::tile_floats();  // fp32 consumers' scratch
  int st = 0;          // the next stage, and
  uint32_t fph = 0;    // the parity of its full barrier's phase (flips at every wrap)
  bool first = true;
  uint32_t seg_phase = 0;  // parity of the row-boundary barriers (TW > 1)
  for (int v = vb; v <= ve && v < V; ++v) {
    int64_t ts, tend;
    seg_bounds(v, ts, tend);
    if (ts >= tend) continue;
    const int r = v % R, hgi = v / R;
    const int kvh = hgi * HG + hl;
    const int64_t c = len_of(v);
    W.begin(p, r, kvh, c, lane);
    bool ok = true;
    for (int64_t cb = ts; cb < tend; cb += CT) {
      ok = mbar_wait(smem_u32(&full_bar[st]), fph, abort);
      if (!__all_sync(FULL, ok)) {
        set_flag(p.err, NP_FLAG_TIMEOUT);
        ok = false;
        break;
      }
      // this warp's slice of the stage: tokens [s0, s1)
      const int nvalid = (int)min((int64_t)CT, tend - cb);
      const int s0 = tw * WS, s1 = min(nvalid, s0 + WS);
      if constexpr (K::kTmap) {
        const uint32_t kst = smem_u32(smem + st * stage_bytes);
        for (int sb = s0; sb < s1; sb += C::ST)
          W.template tile<true>(L, kst, kst + (uint32_t)(stage_bytes / 2), sb, s1, cb, p.qscale,
                                lane);
      } else {
        const float* ks = reinterpret_cast<const float*>(smem + st * stage_bytes);
        for (int k0 = s0; k0 < s1; k0 += C::CT)
          W.consume(ks + (size_t)k0 * HG * D, ks + stage_bytes / 8 + (size_t)k0 * HG * D, hl, HG,
                    min(s1 - k0, C::CT), cb + k0, tile, lane);
      }
      __syncwarp();  // every lane's reads of this stage are done
      if (lane == 0) mbar_arrive(smem_u32(&empty_bar[st]));
      if (++st == stages) {
        st = 0;
        fph ^= 1u;
      }
    }
    if (!ok) return;
    W.finish();
    const bool whole = ts == 0 && tend == c;
    const int slot = first ? 0 : 1;
    first = false;
    float* ent = p.ws_o + (((int64_t)b * 2 + slot) * HG + hl) * (int64_t)StreamWs::entry_floats(D);

    if (TW == 1) {
      if (whole) W.store_out(p, r, kvh, lane);  // the whole row is here: normalise and store
      else W.store_rows(ent, ent + kMmaRows, ent + 2 * kMmaRows, MR, lane, keep);  // cut row
      continue;
    }
    // ---- TW > 1: the head's warps put their states side by side, then each
    // merges a share of the rows (in tw order) and stores them or their
    // partials.
    // Bounded waits: a timed-out pipeline returns instead of waiting here.
    float* my = wstate + (size_t)warp * wstate_entry_floats(MR, D);
    W.store_rows(my, my + wstate_mrp(MR), my + 2 * wstate_mrp(MR), MR, lane);
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&seg_bar[0]));
    if (!__all_sync(FULL, mbar_wait(smem_u32(&seg_bar[0]), seg_phase, abort))) return;
    merge_warp_states<T, D>(p, wstate, hl, HG, TW, tw, MR, Gr, r, kvh, whole, ent, keep, lane);
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&seg_bar[1]));
    // the next boundary's states go to the same place: wait until merged
    if (!__all_sync(FULL, mbar_wait(smem_u32(&seg_bar[1]), seg_phase, abort))) return;
    seg_phase ^= 1u;
  }
}

// One merge task: mma rows row0 .. row0+RPW-1 of kv head hl of the cut
// row v -- head_dim part dh of DH -- over the partials of its covering CTAs
// b0 .. bl in ascending order, in batches of U; each batch is one round of
// loads (lane j: partial j's m and l; every lane: its slice of the part for
// all U partial rows of its RPW mma rows), then a rescale of the running
// state to the batch's max (a fixed order: results are deterministic).
// Every partial the merge reads is finite (an empty one is m = -inf, l = 0,
// o = 0), so the weighted sum runs without branches and its loads all issue
// before the first use.  RPW = 2 when a row group has 16 mma rows (fewer
// tasks per row); DH = 2 when rows are cut many ways: half the head_dim per
// task lets one batch hold 32 partials (one round of loads where a whole
// head_dim would take two).
template <typename T, int D, int G, int RPW, int DH>
struct MergeCfg {
  static constexpr int DL = D / DH / 32;  // dims per lane
  static constexpr int U = 64 / (RPW * DL) < 32 ? 64 / (RPW * DL) : 32;  // partials per batch
  static_assert(DL >= 1 && D % (DH * 32) == 0, "merge slices");
};

template <typename T, int D, int G, int RPW, int DH>
__device__ __forceinline__ void merge_task(const DecodeParams& p, int v, int b0, int bl,
                                           int slot_b0, int row0, int hl, int dh, int lane) {
  constexpr unsigned FULL = 0xffffffffu;
  const int HG = p.head_group;
  constexpr int DL = MergeCfg<T, D, G, RPW, DH>::DL;
  constexpr int U = MergeCfg<T, D, G, RPW, DH>::U;
  const int Q = p.query_len;
  const int Gr = G > 0 ? G : p.q_heads / p.kv_heads;  // G = 0: the group set at run time
  const int MR = Gr * Q;
  const int R = p.rows;
  const int r = v % R, hgi = v / R;
  const int kvh = hgi * HG + hl;
  const int64_t ent_floats = (int64_t)StreamWs::entry_floats(D);
  auto entry = [&](int j) -> const float* {  // CTA j's partial of row v, kv head hl
    return p.ws_o + (((int64_t)j * 2 + (j == b0 ? slot_b0 : 0)) * HG + hl) * ent_floats;
  };
  const int d0 = dh * (D / DH) + lane * DL;
  int rows[RPW];  // this warp's mma rows (a row past MR repeats row0; not stored)
#pragma unroll
  for (int k = 0; k < RPW; ++k) rows[k] = row0 + k < MR ? row0 + k : row0;

  float mm[RPW], lsum[RPW], acc[RPW][DL];
#pragma unroll
  for (int k = 0; k < RPW; ++k) {
    mm[k] = -INFINITY;
    lsum[k] = 0.f;
#pragma unroll
    for (int e2 = 0; e2 < DL; ++e2) acc[k][e2] = 0.f;
  }
  for (int base = b0; base <= bl; base += U) {
    const int nb = min(U, bl - base + 1);
    float mj[RPW], lj[RPW];
#pragma unroll
    for (int k = 0; k < RPW; ++k) {
      mj[k] = -INFINITY;
      lj[k] = 0.f;
    }
    if (lane < nb) {
      const float* e = entry(base + lane);
#pragma unroll
      for (int k = 0; k < RPW; ++k) {
        mj[k] = e[rows[k]];
        lj[k] = e[kMmaRows + rows[k]];
      }
    }
    float ok[RPW][U][DL];
#pragma unroll
    for (int u = 0; u < U; ++u) {  // the batch's partials only (nb is known before any load)
#pragma unroll
      for (int k = 0; k < RPW; ++k) {
        if (u < nb) {
          Storage<float>::template load<DL>(
              entry(base + u) + 2 * kMmaRows + rows[k] * D + d0, ok[k][u]);
        } else {
#pragma unroll
          for (int e2 = 0; e2 < DL; ++e2) ok[k][u][e2] = 0.f;
        }
      }
    }
#pragma unroll
    for (int k = 0; k < RPW; ++k) {
      float bm = mj[k];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) bm = fmaxf(bm, __shfl_xor_sync(FULL, bm, o));
      const float mn = fmaxf(mm[k], bm);
      const float msub = mn == -INFINITY ? 0.f : mn;
      const float sc = ex2(mm[k] - msub);  // mm = -inf: 0 (nothing merged yet)
      const float aj = ex2(mj[k] - msub);  // an empty partial (m = -inf): 0
      float ls = aj * lj[k];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) ls += __shfl_xor_sync(FULL, ls, o);
      lsum[k] = fmaf(lsum[k], sc, ls);
#pragma unroll
      for (int e2 = 0; e2 < DL; ++e2) acc[k][e2] *= sc;
#pragma unroll
      for (int u = 0; u < U; ++u) {  // in CTA order; lanes >= nb hold aj = 0
        const float au = __shfl_sync(FULL, aj, u);
#pragma unroll
        for (int e2 = 0; e2 < DL; ++e2) acc[k][e2] = fmaf(ok[k][u][e2], au, acc[k][e2]);
      }
      mm[k] = mn;
    }
  }
#pragma unroll
  for (int k = 0; k < RPW; ++k) {
    const int row = row0 + k;
    if (row >= MR) break;
    const float inv = lsum[k] > 0.f ? 1.f / lsum[k] : 0.f;
    float ov[DL];
#pragma unroll
    for (int e2 = 0; e2 < DL; ++e2) ov[e2] = acc[k][e2] * inv;
    const int qi = row / Gr, h = row - qi * Gr;
    T* o = static_cast<T*>(p.out) + (((int64_t)r * Q + qi) * p.q_heads + kvh * Gr + h) * D;
    Storage<T>::template store<DL>(o + d0, ov);
  }
}

// Merge of the cut rows.  One block per CTA of the read (one wave).  The
// read left, for each CTA b whose range ends inside a row it began (and so
// cuts it), the descriptor {v, b, bl, slot}: the row, its covering CTAs b ..
// bl and the slot of b's partial.  Every block loads all P descriptors (one
// coalesced round), lists the cut rows in CTA order, and the cut rows' tasks
// -- RPW mma rows of one kv head, one of DH head_dim parts, NT per row, all
// numbered in that order -- are dealt round-robin over the blocks (block c
// takes tasks c, c + P, c + 2P, ..., its warps one each in turn), so every
// SM merges about the same number of tasks whatever the cut rows' lengths
// and however many of them a CTA touches, and a few tasks still spread over
// many SMs.
template <typename T, int D, int G, int RPW, int DH>
__global__ void __launch_bounds__(256 * kMergeRpb) paged_decode_stream_merge_kernel(
    const __grid_constant__ DecodeParams p) {
  const int HG = p.head_group;  // kv heads per row group
  const int c = blockIdx.x;
  const int P = gridDim.x;  // <= kStreamMaxCtas
  const int w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const int lane = threadIdx.x & 31;
  __shared__ int4 s_desc[kStreamMaxCtas];
  __shared__ int s_list[kStreamMaxCtas];  // CTAs that own a cut row, in order
  __shared__ int s_rows;
#if NPK_STREAM_PDL
  asm volatile("griddepcontrol.wait;" ::: "memory");  // the read is complete
#endif
  const int nv = p.rows * (p.kv_heads / HG);
  const int4* desc = reinterpret_cast<const int4*>(p.st_desc);
  for (int b = threadIdx.x; b < P; b += blockDim.x) {
    int4 x = desc[b];
    // a descriptor names a row begun by CTA b and CTAs of this launch, or nothing
    if (!(x.x >= 0 && x.x < nv && x.y == b && x.z >= b && x.z < P && (x.w == 0 || x.w == 1)))
      x.x = -1;
    s_desc[b] = x;
  }
  __syncthreads();
  if (w == 0) {  // list the owners in CTA order (ballots over 32 CTAs at a time)
    int n = 0;
    for (int b0 = 0; b0 < P; b0 += 32) {
      const int b = b0 + lane;
      const bool own = b < P && s_desc[b].x >= 0;
      const unsigned m = __ballot_sync(0xffffffffu, own);
      if (own) s_list[n + __popc(m & ((1u << lane) - 1u))] = b;
      n += __popc(m);
    }
    if (lane == 0) s_rows = n;
  }
  __syncthreads();
  const int Gr = G > 0 ? G : p.q_heads / p.kv_heads;
  const int NT = (Gr * p.query_len + RPW - 1) / RPW * HG * DH;  // tasks per cut row
  const int total = s_rows * NT;
  for (int g = c + w * P; g < total; g += nw * P) {
    const int4 x = s_desc[s_list[g / NT]];
    const int t = g % NT;
    const int hd = t / DH;  // t = hd * DH + part, hd = group * head_group + head
    merge_task<T, D, G, RPW, DH>(p, x.x, x.y, x.z, x.w, (hd / HG) * RPW, hd % HG, t % DH, lane);
  }
}

}  // namespace npk
