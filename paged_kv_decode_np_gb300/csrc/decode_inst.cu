// decode_inst.cu -- instantiates the decode kernel for one storage type and
// head_dim (chosen at compile time: -DNPK_BF16=0/1 -DNPK_D=<head_dim>) and
// for every supported GQA group, behind one launcher function.
#include "decode_fma.cuh"
#include "decode_launch.h"
#include "decode_mma.cuh"
#include "decode_stream.cuh"

#ifndef NPK_BF16
#error "define NPK_BF16"
#endif
#ifndef NPK_D
#error "define NPK_D"
#endif

#if NPK_BF16
using StorageT = __nv_bfloat16;
#define NPK_TNAME bf16
#else
using StorageT = float;
#define NPK_TNAME f32
#endif

#define NPK_CAT3(a, b, c) a##b##c
#define NPK_NAME3(a, b, c) NPK_CAT3(a, b, c)
#define NPK_LAUNCHER NPK_NAME3(decode_, NPK_TNAME, NPK_NAME3(_d, NPK_D, ))

namespace npk {
namespace {

// bf16 pools run on the tensor cores (decode_mma.cuh): through tiled TMA
// boxes when the host built pool maps, else through per-token copies
// (TWO: mma rows past the first 8).  fp32 pools keep full fp32 products on
// the FMA pipes (decode_fma.cuh; TWO: several query tokens, the 8-row
// layout).
template <int G, bool TMAP, bool TWO>
struct Variant {
#if NPK_BF16
  using SM = MmaSmem<NPK_D, G, TMAP>;
  static constexpr auto kernel = paged_decode_mma_kernel<NPK_D, G, TMAP, TWO>;
  static size_t fixed(int) { return 16 + 128 + 1024; }
#else
  using SM = FmaSplitSmem<NPK_D, G, TWO>;
  static constexpr auto kernel = paged_decode_fma_kernel<NPK_D, G, TWO>;
  static size_t fixed(int warps) { return SM::tiles_bytes(warps) + 16 + 128; }
#endif
};

template <int G, bool TMAP, bool TWO>
np_status launch_variant(DecodeLaunch& L, DecodeParams& p) {
  using V = Variant<G, TMAP, TWO>;
  using SM = typename V::SM;
  const int warps = L.head_group * L.token_warps;
  const size_t fixed = V::fixed(warps);
  const size_t sb = SM::stage_bytes(L.head_group);
  if (L.smem_budget <= fixed) return NP_ERR_UNSUPPORTED;
  size_t stages = (L.smem_budget - fixed) / (sb + 16);
  if (stages > 8) stages = 8;
  if (stages < 2) return NP_ERR_UNSUPPORTED;
  while (stages > 2 && SM::total(L.head_group, (int)stages, warps) > L.smem_budget) --stages;
  const size_t smem = SM::total(L.head_group, (int)stages, warps);
  if (smem > L.smem_budget) return NP_ERR_UNSUPPORTED;
  p.stages = (int)stages;
  L.stages = (int)stages;
  L.smem_bytes = smem;

  auto kern = V::kernel;
  // The opt-in shared-memory limit is a per-device function attribute.
  static unsigned long long configured = 0;  // bit d: done on device d
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return NP_ERR_CUDA;
  if (dev >= 64 || !((__atomic_load_n(&configured, __ATOMIC_ACQUIRE) >> dev) & 1ull)) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)L.smem_budget) != cudaSuccess)
      return NP_ERR_CUDA;
    if (dev < 64) __atomic_fetch_or(&configured, 1ull << dev, __ATOMIC_ACQ_REL);
  }
  dim3 grid(L.splits, L.rows, L.head_groups);
  kern<<<grid, 32 * (warps + 1), smem, L.stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? NP_OK : NP_ERR_CUDA;
}

#if (NPK_BF16 && NPK_D % 64 == 0) || (!NPK_BF16 && NPK_D % 32 == 0)
#define NPK_HAS_STREAM 1
#ifndef NPK_MERGE_RPW4
#define NPK_MERGE_RPW4 1
#endif

// The balanced streamed read: grid = L.splits CTAs (one per SM), HG kv heads
// per CTA, the virtual-row prefix in shared memory after the ring.
template <int G, bool TWO>
np_status launch_stream(DecodeLaunch& L, DecodeParams& p) {
  using SS = StreamSmem<StorageT, NPK_D, G, TWO>;
  const int hg = p.head_group;  // kv heads per CTA
  const int vrows = p.rows * (p.kv_heads / hg);
  // static shared memory of the kernel (scan scratch) comes off the budget
  const size_t budget = L.smem_budget - 4096;
  // a ring of up to 192 KB in flight (fewer, larger stages with more heads);
  // when TW > 1 consumer warps per head leave no room for two stages next to
  // their row-boundary states, half as many warps per head read (a stage of
  // fewer tokens still divides the block table's 32-block windows)
  size_t stages = 0;
  int tw = p.token_warps;
  const int sl = p.stage_slices;  // K::CT-token pieces per warp and stage
  const int mr = L.group * p.query_len;  // (query token, head) rows per kv head
  for (;;) {
    const size_t sb = SS::stage_bytes(hg, tw * sl);
    stages = (196608 / sb) < 2 ? 2 : (196608 / sb) > 32 ? 32 : 196608 / sb;
    while (stages >= 2 && SS::total(hg, tw * sl, (int)stages, vrows, tw, hg * tw, mr) > budget)
      --stages;
    if (stages >= 2 || tw == 1) break;
    tw = tw % 2 == 0 ? tw / 2 : 1;
  }
  if (stages < 2) return NP_ERR_UNSUPPORTED;
  p.token_warps = tw;
  L.token_warps = tw;
  const size_t smem = SS::total(hg, tw * sl, (int)stages, vrows, tw, hg * tw, mr);
  p.stages = (int)stages;
  L.stages = (int)stages;
  L.smem_bytes = smem;
  // several warps per kv head: the build with their row-end merges
  const int multi = tw > 1 ? 1 : 0;
  auto kern = multi ? paged_decode_stream_kernel<StorageT, NPK_D, G, TWO, true>
                    : paged_decode_stream_kernel<StorageT, NPK_D, G, TWO, false>;
  static unsigned long long configured[2] = {0, 0};  // bit d: attribute set on device d
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return NP_ERR_CUDA;
  if (dev >= 64 ||
      !((__atomic_load_n(&configured[multi], __ATOMIC_ACQUIRE) >> dev) & 1ull)) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)budget) !=
        cudaSuccess)
      return NP_ERR_CUDA;
    if (dev < 64) __atomic_fetch_or(&configured[multi], 1ull << dev, __ATOMIC_ACQ_REL);
  }
  kern<<<L.splits, 32 * (8 + 1), smem, L.stream>>>(p);
  if (cudaGetLastError() != cudaSuccess) return NP_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(L.splits, 1);  // one block per CTA of the read
  cfg.blockDim = dim3(256 * kMergeRpb);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = L.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = NPK_STREAM_PDL;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // Merge tasks: two mma rows each when a row group has 16 (four when the
  // cut rows' tasks would otherwise outnumber the merge's warps and a row is
  // cut into at most ~4 pieces, one batch of 4 partials); half the head_dim
  // each when the rows are likely cut into more than 16 pieces (more CTAs
  // than 16 per virtual row), so that one round of loads covers a row's
  // partials.
  cudaError_t rc = cudaErrorInvalidValue;
  bool done = false;
#if NPK_MERGE_RPW4
  if (mr >= 16) {
    const int64_t cut_rows = vrows < L.splits ? vrows : L.splits;
    const int64_t tasks2 = cut_rows * (mr / 2) * hg;
    const int64_t warps = (int64_t)L.splits * (256 * kMergeRpb / 32);
    if (tasks2 > warps && L.splits <= 3 * vrows) {
      rc = cudaLaunchKernelEx(&cfg, paged_decode_stream_merge_kernel<StorageT, NPK_D, G, 4, 1>, p);
      done = true;
    }
  }
#endif
  if constexpr (NPK_D >= 64 && NPK_MERGE_DH2) {
    if (mr < 16 && 16 * vrows < L.splits) {
      rc = cudaLaunchKernelEx(&cfg, paged_decode_stream_merge_kernel<StorageT, NPK_D, G, 1, 2>, p);
      done = true;
    }
  }
  if (!done)
    rc = mr >= 16
             ? cudaLaunchKernelEx(&cfg, paged_decode_stream_merge_kernel<StorageT, NPK_D, G, 2, 1>, p)
             : cudaLaunchKernelEx(&cfg, paged_decode_stream_merge_kernel<StorageT, NPK_D, G, 1, 1>, p);
  if (rc != cudaSuccess) return NP_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? NP_OK : NP_ERR_CUDA;
}
#endif

// bf16 (G = 0: the group is read at run time, any g with g * query_len <=
// 16): TWO when the (query token, head) rows spill past the first 8 mma rows.
// fp32: several query tokens only on the balanced read, at most 8 rows
// (host-checked).
template <int G>
np_status launch_one(DecodeLaunch& L, DecodeParams& p) {
#if defined(NPK_HAS_STREAM) && NPK_BF16
  if (L.streamed)
    return L.group * p.query_len > 8 ? launch_stream<G, true>(L, p)
                                     : launch_stream<G, false>(L, p);
#elif defined(NPK_HAS_STREAM)
  if (L.streamed) {  // fp32: several query tokens as (query token, head) rows, up to 8
    if constexpr (G <= 4)
      if (p.query_len > 1) return launch_stream<G, true>(L, p);
    return launch_stream<G, false>(L, p);
  }
#endif
  if (L.streamed) return NP_ERR_UNSUPPORTED;
#if NPK_BF16
  const bool two = L.group * p.query_len > 8;
#if NPK_D % 64 == 0
  if (p.use_tmap)
    return two ? launch_variant<G, true, true>(L, p) : launch_variant<G, true, false>(L, p);
#endif
  p.use_tmap = 0;
  return two ? launch_variant<G, false, true>(L, p) : launch_variant<G, false, false>(L, p);
#else
  p.use_tmap = 0;
  // several query tokens: (query token, head) rows, up to 8, group at run time
  return p.query_len > 1 ? launch_variant<0, false, true>(L, p)
                         : launch_variant<G, false, false>(L, p);
#endif
}

}  // namespace

np_status NPK_LAUNCHER(DecodeLaunch& L, DecodeParams& p) {
#if NPK_BF16
  return launch_one<0>(L, p);  // the tensor-core warps take the group at run time
#else
  switch (L.group) {
    case 1: return launch_one<1>(L, p);
    case 2: return launch_one<2>(L, p);
    case 4: return launch_one<4>(L, p);
    case 5: return launch_one<5>(L, p);
    case 8: return launch_one<8>(L, p);
    default:
      // other groups up to 8: the FMA warp's 8-row layout with the group read
      // at run time (host-checked: g * query_len <= 8)
      if (L.group > 8) return NP_ERR_UNSUPPORTED;
#ifdef NPK_HAS_STREAM
      if (L.streamed) return launch_stream<0, true>(L, p);
#endif
      if (L.streamed) return NP_ERR_UNSUPPORTED;
      p.use_tmap = 0;
      return launch_variant<0, false, true>(L, p);
  }
#endif
}

}  // namespace npk
