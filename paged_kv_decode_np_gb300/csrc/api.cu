// api.cu -- the C ABI of libnp_paged.so (declared in include/np_paged.h):
// argument validation, split planning from static shapes, and launches.
// Nothing here allocates, synchronises or reads device memory.
#include <limits.h>
#include <math.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include <cudaTypedefs.h>  // PFN_cuTensorMapEncodeTiled_v12000

#include "decode_kernel.cuh"
#include "decode_launch.h"
#include "decode_stream.cuh"
#include "np_paged.h"

#ifndef NPK_SPLIT_BYTES
#define NPK_SPLIT_BYTES (2ll << 20)  // K+V bytes one split should read
#endif

#ifndef NPK_SMEM_BUDGET
#define NPK_SMEM_BUDGET 0  // 0: the device's opt-in maximum per block
#endif

namespace {

using npk::DecodeLaunch;
using npk::DecodeParams;

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int elem_size(np_dtype d) { return d == NP_F32 ? 4 : (d == NP_BF16 ? 2 : 0); }

bool head_dim_supported(int32_t d) {
  return d == 16 || d == 32 || d == 64 || d == 128 || d == 256;
}

// GQA group g = q_heads / kv_heads: any g up to 16 on bf16 pools (the
// tensor-core warps take it at run time; g * query_len <= 16 is checked with
// the query tokens), up to 8 on fp32 pools (the FMA warp holds 8 rows;
// groups outside {1, 2, 4, 5, 8} take its run-time-group layout).
bool group_supported(np_dtype dtype, int32_t g) {
  return g >= 1 && g <= (dtype == NP_BF16 ? 16 : 8);
}

// a*b*... without int64 overflow; false on overflow or negative input
bool mul_ok(int64_t a, int64_t b, int64_t* out) {
  if (a < 0 || b < 0) return false;
  if (a != 0 && b > INT64_MAX / a) return false;
  *out = a * b;
  return true;
}

// kv heads per CTA: the largest divisor of kv_heads that is <= 8
int head_group_of(int32_t kv_heads) {
  for (int hg = 8; hg >= 1; --hg)
    if (kv_heads % hg == 0) return hg;
  return 1;
}

struct DeviceInfo {
  std::atomic<int> sms{0};
  std::atomic<int> smem_optin{0};
};
DeviceInfo g_dev[64];

np_status device_info(int* sms, int* smem) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return NP_ERR_CUDA;
  DeviceInfo* di = dev < 64 ? &g_dev[dev] : nullptr;
  int s = di ? di->sms.load() : 0, m = di ? di->smem_optin.load() : 0;
  if (s == 0 || m == 0) {
    if (cudaDeviceGetAttribute(&s, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&m, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
      return NP_ERR_CUDA;
    if (di) {
      di->sms.store(s);
      di->smem_optin.store(m);
    }
  }
  *sms = s;
  *smem = m;
  return NP_OK;
}

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Consumer warps per kv head of the balanced streamed read (TW): up to
// 8 / HG, each taking ct0 tokens of every stage (ct0: the consumer warp's
// chunk, 1024 / head_dim fp32 rows or the mma chunk), so that a stage holds
// TW * ct0 tokens and the per-stage costs of the producer (barriers, table
// lookups, copy issue) are paid once per TW * ct0 tokens.  A stage must not
// straddle two 32-block windows of the block table: TW * ct0 divides
// 32 * block_size.  HG = 4 keeps one warp per head when built with
// NPK_STREAM_TW4=0.
#ifndef NPK_STREAM_TW4
#define NPK_STREAM_TW4 0
#endif
#ifndef NPK_STREAM_TWMAX
#define NPK_STREAM_TWMAX 8
#endif
// One- and two-head groups: four consumer warps (two pieces of each stage
// apiece), so that their row-end states leave room for three 64 KB stages.
#ifndef NPK_STREAM_NCW4
#define NPK_STREAM_NCW4 1
#endif
int stream_chunk_tokens(np_dtype dtype, int32_t head_dim) {
  return dtype == NP_BF16 ? npk::mma_chunk_tokens(head_dim) : 1024 / head_dim;
}
int stream_token_warps(np_dtype dtype, int32_t head_dim, int hg, int32_t block_size) {
  if (hg == 4 && !NPK_STREAM_TW4) return 1;
  const int ct0 = stream_chunk_tokens(dtype, head_dim);
  int tw = (NPK_STREAM_NCW4 && hg <= 2 ? 4 : npk::kMaxConsumerWarps) / hg;
  if (tw > NPK_STREAM_TWMAX) tw = NPK_STREAM_TWMAX;
  while (tw > 1 && ((int64_t)32 * block_size) % ((int64_t)ct0 * tw) != 0) --tw;
  return tw;
}

// K::CT-token pieces each consumer warp takes per stage (SL): with fewer than
// 8 consumer warps (HG * TW < 8, e.g. four kv heads with one warp each) a
// stage holds 8 / (HG * TW) pieces per warp, so that it still moves about
// 64 KB per producer iteration; SL * TW * ct0 divides 32 * block_size.
// Built with NPK_STREAM_SLICES=0: one piece.
#ifndef NPK_STREAM_SLICES
#define NPK_STREAM_SLICES 1
#endif
int stream_stage_slices(np_dtype dtype, int32_t head_dim, int hg, int tw, int32_t block_size) {
  if (!NPK_STREAM_SLICES) return 1;
  const int ct0 = stream_chunk_tokens(dtype, head_dim);
  int sl = npk::kMaxConsumerWarps / (hg * tw);
  if (sl < 1) sl = 1;
  while (sl > 1 && ((int64_t)32 * block_size) % ((int64_t)ct0 * tw * sl) != 0) --sl;
  return sl;
}

// Tokens per tiled TMA box of the bf16 read: the largest power of two that
// divides the block size, at most a stage's tokens.
int box_tokens_for(int32_t block_size, int32_t head_dim) {
  const int ct = npk::mma_chunk_tokens(head_dim);
  int bt = 1;
  while (bt < ct && block_size % (bt * 2) == 0) bt *= 2;
  return bt;
}

// Shapes the balanced streamed read (num_splits == 0) handles: bf16 pools
// with head_dim a multiple of 64 (tiled TMA boxes of box_tokens x HG heads
// starting on 1024-byte swizzle boundaries: box_tokens * HG a multiple of 8)
// or fp32 pools with head_dim a multiple of 32, at most kStreamMaxVRows
// (row, head group) pairs, contexts that fit int32.  HG is the largest
// divisor of kv_heads up to 8.
bool stream_ok(np_dtype dtype, int32_t head_dim, int32_t kv_heads, int32_t rows,
               int32_t max_blocks_per_row, int32_t block_size) {
  const int hg = head_group_of(kv_heads);
  const bool dim_ok = dtype == NP_BF16 ? head_dim % 64 == 0 : head_dim % 32 == 0;
  return dim_ok && head_dim <= 256 &&
         (dtype != NP_BF16 || (box_tokens_for(block_size, head_dim) * hg) % 8 == 0) &&
         (int64_t)rows * (kv_heads / hg) <= npk::kStreamMaxVRows &&
         (int64_t)max_blocks_per_row * block_size <= INT32_MAX;
}

// ---- tiled TMA maps of the pools (bf16, head_dim a multiple of 64)
// The driver's encoder is reached through the runtime (no libcuda link).
PFN_cuTensorMapEncodeTiled_v12000 tmap_encoder() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// L2 promotion of the pool maps' requests (CUtensorMapL2promotion).
#ifndef NPK_TMAP_L2_PROMO
#define NPK_TMAP_L2_PROMO CU_TENSOR_MAP_L2_PROMOTION_L2_256B
#endif

// Map of one pool as a 4-D tensor (64 dims, slot, kv head, 64-dim slab):
// the dimensions are listed in the order a box lands in shared memory, not
// by stride, so that one box {64, box_tokens, head_group, head_dim/64}
// arrives as [slab][head][token][64 dims] -- each head's tokens in
// consecutive 128-byte rows (128-byte swizzle) -- and one copy per box
// brings every slab of its tokens.  Returns false if the driver refuses.
bool encode_pool_map(CUtensorMap* m, const void* pool, int64_t slots, int32_t kv_heads,
                     int32_t head_dim, int box_tokens, int head_group) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tmap_encoder();
  if (!enc) return false;
  cuuint64_t dims[4] = {64u, (cuuint64_t)slots, (cuuint64_t)kv_heads,
                        (cuuint64_t)(head_dim / 64)};
  cuuint64_t strides[3] = {(cuuint64_t)kv_heads * head_dim * 2, (cuuint64_t)head_dim * 2, 128u};
  cuuint32_t box[4] = {64u, (cuuint32_t)box_tokens, (cuuint32_t)head_group,
                       (cuuint32_t)(head_dim / 64)};
  cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
  CUresult rc = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(pool), dims, strides,
                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    NPK_TMAP_L2_PROMO, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return rc == CUDA_SUCCESS;
}

// Small per-thread cache: the same pools are read step after step.
struct MapKey {
  const void* k;
  const void* v;
  int64_t slots;
  int32_t kv_heads, head_dim, box_tokens, head_group, device;
  bool operator==(const MapKey& o) const {
    return k == o.k && v == o.v && slots == o.slots && kv_heads == o.kv_heads &&
           head_dim == o.head_dim && box_tokens == o.box_tokens && head_group == o.head_group &&
           device == o.device;
  }
};
struct MapEntry {
  MapKey key;
  CUtensorMap mk, mv;
  bool ok;
  bool used;
};

bool pool_maps(DecodeParams& p, const void* k, const void* v, int64_t slots, int32_t kv_heads,
               int32_t head_dim, int box_tokens, int head_group) {
  thread_local MapEntry cache[4] = {};
  thread_local int next = 0;
  int dev = 0;
  cudaGetDevice(&dev);
  MapKey key{k, v, slots, kv_heads, head_dim, box_tokens, head_group, dev};
  for (auto& e : cache) {
    if (e.used && e.key == key) {
      p.tm_k = e.mk;
      p.tm_v = e.mv;
      return e.ok;
    }
  }
  MapEntry& e = cache[next];
  next = (next + 1) % 4;
  e.key = key;
  e.used = true;
  e.ok = encode_pool_map(&e.mk, k, slots, kv_heads, head_dim, box_tokens, head_group) &&
         encode_pool_map(&e.mv, v, slots, kv_heads, head_dim, box_tokens, head_group);
  p.tm_k = e.mk;
  p.tm_v = e.mv;
  return e.ok;
}

npk::DecodeLauncher launcher_for(np_dtype dt, int32_t d) {
  if (dt == NP_F32) {
    switch (d) {
      case 16: return npk::decode_f32_d16;
      case 32: return npk::decode_f32_d32;
      case 64: return npk::decode_f32_d64;
      case 128: return npk::decode_f32_d128;
      case 256: return npk::decode_f32_d256;
    }
  } else if (dt == NP_BF16) {
    switch (d) {
      case 16: return npk::decode_bf16_d16;
      case 32: return npk::decode_bf16_d32;
      case 64: return npk::decode_bf16_d64;
      case 128: return npk::decode_bf16_d128;
      case 256: return npk::decode_bf16_d256;
    }
  }
  return nullptr;
}

}  // namespace

extern "C" {

const char* np_status_string(np_status s) {
  switch (s) {
    case NP_OK: return "NP_OK";
    case NP_ERR_INVALID_ARG: return "NP_ERR_INVALID_ARG";
    case NP_ERR_UNSUPPORTED: return "NP_ERR_UNSUPPORTED";
    case NP_ERR_WORKSPACE: return "NP_ERR_WORKSPACE";
    case NP_ERR_OUT_OF_RANGE: return "NP_ERR_OUT_OF_RANGE";
    case NP_ERR_CUDA: return "NP_ERR_CUDA";
  }
  return "NP_ERR_UNKNOWN";
}

int32_t np_abi_version(void) { return NP_ABI_VERSION; }

np_status np_kv_append(void* k_pool, void* v_pool, np_dtype dtype, int64_t num_blocks,
                       int32_t block_size, int32_t kv_heads, int32_t head_dim,
                       const void* k_new, const void* v_new, const int64_t* slot_mapping,
                       int32_t num_tokens, int32_t* err_word, np_stream_t stream) {
  const int es = elem_size(dtype);
  if (es == 0) return NP_ERR_UNSUPPORTED;
  if (num_blocks <= 0 || block_size <= 0 || kv_heads <= 0 || head_dim <= 0 || num_tokens < 0)
    return NP_ERR_INVALID_ARG;
  int64_t row_bytes = 0, slots = 0, pool_bytes = 0;
  if (!mul_ok((int64_t)kv_heads * es, head_dim, &row_bytes) ||
      !mul_ok(num_blocks, block_size, &slots) || !mul_ok(slots, row_bytes, &pool_bytes))
    return NP_ERR_OUT_OF_RANGE;
  if (row_bytes % 16 != 0) return NP_ERR_UNSUPPORTED;
  if (num_tokens == 0) return NP_OK;
  if (!k_pool || !v_pool || !k_new || !v_new || !slot_mapping) return NP_ERR_INVALID_ARG;
  if (!aligned(k_pool, 16) || !aligned(v_pool, 16) || !aligned(k_new, 16) ||
      !aligned(v_new, 16) || !aligned(slot_mapping, 8) || (err_word && !aligned(err_word, 4)))
    return NP_ERR_INVALID_ARG;
  return npk::launch_append(k_pool, v_pool, slots, row_bytes, k_new, v_new, slot_mapping,
                            num_tokens, err_word, reinterpret_cast<cudaStream_t>(stream));
}

int64_t np_paged_decode_split_len(int32_t block_size, int32_t max_blocks_per_row,
                                  int32_t num_splits) {
  if (block_size <= 0 || max_blocks_per_row <= 0 || num_splits <= 0) return -1;
  const int64_t cap = (int64_t)max_blocks_per_row * block_size;
  const int64_t align = block_size > 64 ? block_size : 64;
  int64_t sl = (cap + num_splits - 1) / num_splits;
  sl = (sl + align - 1) / align * align;
  return sl;
}

np_status np_paged_decode_plan(int32_t rows, int32_t q_heads, int32_t kv_heads,
                               int32_t head_dim, int32_t block_size,
                               int32_t max_blocks_per_row, np_dtype dtype, int32_t num_sms,
                               int32_t* num_splits) {
  const int es = elem_size(dtype);
  if (!num_splits) return NP_ERR_INVALID_ARG;
  if (es == 0) return NP_ERR_UNSUPPORTED;
  if (rows < 0 || q_heads <= 0 || kv_heads <= 0 || q_heads % kv_heads != 0 || head_dim <= 0 ||
      block_size <= 0 || max_blocks_per_row <= 0)
    return NP_ERR_INVALID_ARG;
  if (stream_ok(dtype, head_dim, kv_heads, rows, max_blocks_per_row, block_size)) {
    *num_splits = 0;  // the balanced streamed read
    return NP_OK;
  }
  if (num_sms <= 0) {
    int smem = 0;
    np_status st = device_info(&num_sms, &smem);
    if (st != NP_OK) return st;
  }
  const int g = q_heads / kv_heads;
  const int hg = head_group_of(kv_heads);
  const int64_t units = (int64_t)rows * (kv_heads / hg);
  const int64_t cap = (int64_t)max_blocks_per_row * block_size;
  // Tokens per split: about 2 MB of K+V per CTA, and at least 128x the
  // partial result it writes (so partials + reduce stay ~1% of the traffic).
  const int64_t tok_bytes = 2ll * hg * head_dim * es;
  int64_t sl = NPK_SPLIT_BYTES / tok_bytes;
  const int64_t sl_partial = 256ll * g / es;
  if (sl < sl_partial) sl = sl_partial;
  sl = (sl + 63) / 64 * 64;
  int64_t s = (cap + sl - 1) / sl;
  // Few, short rows: split finer so at least ~2 CTAs per SM exist.
  while (units * s < 2ll * num_sms && sl > 64) {
    sl = (sl / 2 + 63) / 64 * 64;
    s = (cap + sl - 1) / sl;
  }
  if (s < 1) s = 1;
  if (s > 65535) s = 65535;
  *num_splits = (int32_t)s;
  return NP_OK;
}

size_t np_paged_decode_workspace_bytes(int32_t rows, int32_t q_heads, int32_t head_dim,
                                       int32_t num_splits) {
  if (rows <= 0 || q_heads <= 0 || head_dim <= 0 || num_splits < 0) return 0;
  if (num_splits == 0)  // balanced streamed read
    return round_up(npk::StreamWs::bytes(head_dim), 256);
  if (num_splits == 1) return 0;
  const size_t units = (size_t)rows * q_heads * num_splits;
  return round_up(units * head_dim * sizeof(float), 256) + round_up(units * sizeof(float), 256);
}

}  // extern "C"

namespace {

// The read, optionally with the fused append (k_new/v_new/slot_mapping non-null).
np_status decode_impl(void* out, const void* q, const void* k_pool, const void* v_pool,
                      np_dtype dtype, int64_t num_blocks, int32_t block_size, int32_t kv_heads,
                      int32_t head_dim, const int32_t* block_tables, int32_t max_blocks_per_row,
                      const int32_t* context_lens, int32_t rows, int32_t query_len,
                      int32_t q_heads, float scale, int32_t num_splits, void* workspace,
                      size_t workspace_bytes, int32_t* err_word, np_stream_t stream,
                      const void* k_new, const void* v_new, const int64_t* slot_mapping) {
  const int es = elem_size(dtype);
  if (es == 0) return NP_ERR_UNSUPPORTED;
  if (rows < 0 || query_len <= 0 || q_heads <= 0 || kv_heads <= 0 || q_heads % kv_heads != 0 ||
      num_blocks <= 0 || block_size <= 0 || max_blocks_per_row <= 0 || num_splits < 0 ||
      num_splits > 65535 || !isfinite(scale))
    return NP_ERR_INVALID_ARG;
  if (!head_dim_supported(head_dim)) return NP_ERR_UNSUPPORTED;
  if (!group_supported(dtype, q_heads / kv_heads)) return NP_ERR_UNSUPPORTED;
  // several query tokens: (query token, head) rows of a group <= 16 on bf16
  // pools, <= 8 on fp32 pools
  if (query_len > 1) {
    const int64_t mrows = (int64_t)(q_heads / kv_heads) * query_len;
    if (mrows > (dtype == NP_BF16 ? 16 : 8)) return NP_ERR_UNSUPPORTED;
  }
  // the fp32 warps keep token positions in int32
  if (dtype == NP_F32 && (int64_t)max_blocks_per_row * block_size > INT32_MAX)
    return NP_ERR_UNSUPPORTED;
  int64_t slots = 0, pool_elems = 0, pool_bytes = 0, tab = 0;
  if (!mul_ok(num_blocks, block_size, &slots) ||
      !mul_ok(slots, (int64_t)kv_heads * head_dim, &pool_elems) ||
      !mul_ok(pool_elems, es, &pool_bytes) || !mul_ok(rows, max_blocks_per_row, &tab) ||
      !mul_ok(max_blocks_per_row, block_size, &tab))
    return NP_ERR_OUT_OF_RANGE;
  if (rows > 65535) return NP_ERR_UNSUPPORTED;  // grid.y
  if (rows == 0) return NP_OK;
  if (!q || !k_pool || !v_pool || !block_tables || !context_lens) return NP_ERR_INVALID_ARG;
  if (num_splits <= 1 && !out) return NP_ERR_INVALID_ARG;
  const bool streamed = num_splits == 0;
  if (streamed && !stream_ok(dtype, head_dim, kv_heads, rows, max_blocks_per_row, block_size))
    return NP_ERR_UNSUPPORTED;
  if (!aligned(q, 16) || !aligned(k_pool, 16) || !aligned(v_pool, 16) ||
      (out && !aligned(out, 16)) || !aligned(block_tables, 4) || !aligned(context_lens, 4) ||
      (err_word && !aligned(err_word, 4)))
    return NP_ERR_INVALID_ARG;
  float* ws_o = nullptr;
  float* ws_lse = nullptr;
  int32_t* st_desc = nullptr;
  if (streamed) {
    const size_t need = npk::StreamWs::bytes(head_dim);
    if (!workspace || workspace_bytes < need || !aligned(workspace, 256)) return NP_ERR_WORKSPACE;
    ws_o = static_cast<float*>(workspace);
    st_desc = reinterpret_cast<int32_t*>(static_cast<char*>(workspace) +
                                         npk::StreamWs::parts_bytes(head_dim));
  } else if (num_splits > 1) {
    const int32_t units_rows = rows * query_len;  // rows of the partial layout
    const size_t need =
        np_paged_decode_workspace_bytes(units_rows, q_heads, head_dim, num_splits);
    if (!workspace || workspace_bytes < need || !aligned(workspace, 256)) return NP_ERR_WORKSPACE;
    ws_o = static_cast<float*>(workspace);
    ws_lse = reinterpret_cast<float*>(
        static_cast<char*>(workspace) +
        round_up((size_t)units_rows * q_heads * num_splits * head_dim * sizeof(float), 256));
  }
  int sms = 0, smem_optin = 0;
  np_status st = device_info(&sms, &smem_optin);
  if (st != NP_OK) return st;

  const int hg = head_group_of(kv_heads);
  DecodeParams p{};
  p.out = out;
  p.ws_o = ws_o;
  p.ws_lse = ws_lse;
  p.q = q;
  p.k_pool = k_pool;
  p.v_pool = v_pool;
  p.block_tables = block_tables;
  p.context_lens = context_lens;
  p.err = err_word;
  p.num_blocks = num_blocks;
  p.split_len =
      streamed ? 0 : np_paged_decode_split_len(block_size, max_blocks_per_row, num_splits);
  p.block_size = block_size;
  p.kv_heads = kv_heads;
  p.head_group = hg;
  p.token_warps =
      streamed ? stream_token_warps(dtype, head_dim, hg, block_size) : npk::kMaxConsumerWarps / hg;
  p.stage_slices =
      streamed ? stream_stage_slices(dtype, head_dim, hg, p.token_warps, block_size) : 1;
  p.max_blocks_per_row = max_blocks_per_row;
  p.q_heads = q_heads;
  p.num_splits = num_splits;
  p.stages = 0;
  p.qscale = scale * 1.4426950408889634f;  // log2(e)
  p.k_new = k_new;
  p.v_new = v_new;
  p.slot_mapping = slot_mapping;
  p.query_len = query_len;
  p.rows = rows;
  p.st_desc = st_desc;
  // bf16 pools with head_dim a multiple of 64 stage K/V through tiled TMA
  // boxes of box_tokens tokens: the largest power of two dividing the block
  // size, at most the stage's token count, with box_tokens * head_group a
  // multiple of 8 (each box then starts on a 1024-byte swizzle boundary) and
  // slot coordinates in int32.
  p.use_tmap = 0;
  p.box_tokens = 1;
  if (dtype == NP_BF16 && head_dim % 64 == 0 && slots <= INT32_MAX) {
    const int bt = box_tokens_for(block_size, head_dim);  // a box never exceeds a stage
    if ((bt * hg) % 8 == 0 &&
        pool_maps(p, k_pool, v_pool, slots, kv_heads, head_dim, bt, hg)) {
      p.use_tmap = 1;
      p.box_tokens = bt;
    }
  }

  DecodeLaunch L{};
  L.params = &p;
  L.group = q_heads / kv_heads;
  L.head_group = hg;
  L.token_warps = p.token_warps;
  L.rows = rows;
  L.splits = num_splits;
  L.head_groups = kv_heads / hg;
  L.streamed = streamed;
  if (streamed) {
    // bf16: the streamed read stages through the TMA maps
    if (dtype == NP_BF16 && !p.use_tmap) return NP_ERR_UNSUPPORTED;
    L.splits = sms < npk::kStreamMaxCtas ? sms : npk::kStreamMaxCtas;
  }
  L.smem_budget = NPK_SMEM_BUDGET > 0 && NPK_SMEM_BUDGET < smem_optin ? NPK_SMEM_BUDGET
                                                                      : (size_t)smem_optin;
  L.stream = reinterpret_cast<cudaStream_t>(stream);
  npk::DecodeLauncher fn = launcher_for(dtype, head_dim);
  if (!fn) return NP_ERR_UNSUPPORTED;
  return fn(L, p);
}

}  // namespace

extern "C" {

np_status np_paged_decode(void* out, const void* q, const void* k_pool, const void* v_pool,
                          np_dtype dtype, int64_t num_blocks, int32_t block_size,
                          int32_t kv_heads, int32_t head_dim, const int32_t* block_tables,
                          int32_t max_blocks_per_row, const int32_t* context_lens, int32_t rows,
                          int32_t query_len, int32_t q_heads, float scale, int32_t num_splits,
                          void* workspace, size_t workspace_bytes, int32_t* err_word,
                          np_stream_t stream) {
  return decode_impl(out, q, k_pool, v_pool, dtype, num_blocks, block_size, kv_heads, head_dim,
                     block_tables, max_blocks_per_row, context_lens, rows, query_len, q_heads,
                     scale, num_splits, workspace, workspace_bytes, err_word, stream, nullptr,
                     nullptr, nullptr);
}

np_status np_paged_append_decode(void* out, const void* q, const void* k_new, const void* v_new,
                                 const int64_t* slot_mapping, void* k_pool, void* v_pool,
                                 np_dtype dtype, int64_t num_blocks, int32_t block_size,
                                 int32_t kv_heads, int32_t head_dim,
                                 const int32_t* block_tables, int32_t max_blocks_per_row,
                                 const int32_t* context_lens, int32_t rows, int32_t query_len,
                                 int32_t q_heads, float scale, int32_t num_splits,
                                 void* workspace, size_t workspace_bytes, int32_t* err_word,
                                 np_stream_t stream) {
  if (rows > 0) {
    if (!k_new || !v_new || !slot_mapping) return NP_ERR_INVALID_ARG;
    if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(slot_mapping, 8))
      return NP_ERR_INVALID_ARG;
  }
  return decode_impl(out, q, k_pool, v_pool, dtype, num_blocks, block_size, kv_heads, head_dim,
                     block_tables, max_blocks_per_row, context_lens, rows, query_len, q_heads,
                     scale, num_splits, workspace, workspace_bytes, err_word, stream, k_new,
                     v_new, slot_mapping);
}

np_status np_paged_decode_reduce(void* out, np_dtype out_dtype, const void* workspace,
                                 size_t workspace_bytes, int32_t rows, int32_t q_heads,
                                 int32_t head_dim, int32_t num_splits, np_stream_t stream) {
  if (elem_size(out_dtype) == 0) return NP_ERR_UNSUPPORTED;
  if (rows < 0 || q_heads <= 0 || num_splits <= 0 || num_splits > 65535)
    return NP_ERR_INVALID_ARG;
  if (!head_dim_supported(head_dim)) return NP_ERR_UNSUPPORTED;
  if (rows == 0) return NP_OK;
  if (!out || !aligned(out, 16)) return NP_ERR_INVALID_ARG;
  if (num_splits == 1) return NP_ERR_INVALID_ARG;  // nothing to merge: decode wrote out
  const size_t need = np_paged_decode_workspace_bytes(rows, q_heads, head_dim, num_splits);
  if (!workspace || workspace_bytes < need || !aligned(workspace, 256)) return NP_ERR_WORKSPACE;
  const float* ws_o = static_cast<const float*>(workspace);
  const float* ws_lse = reinterpret_cast<const float*>(
      static_cast<const char*>(workspace) +
      round_up((size_t)rows * q_heads * num_splits * head_dim * sizeof(float), 256));
  return npk::launch_reduce(out, out_dtype, ws_o, ws_lse, rows, q_heads, head_dim, num_splits,
                            reinterpret_cast<cudaStream_t>(stream));
}

np_status np_selftest_bounded_wait(int32_t* err_word, int64_t limit_cycles, np_stream_t stream) {
  if (!err_word || !aligned(err_word, 4) || limit_cycles < 1 ||
      limit_cycles > npk::kWaitLimitCycles)
    return NP_ERR_INVALID_ARG;
  return npk::launch_bounded_wait_check(err_word, limit_cycles,
                                        reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"
