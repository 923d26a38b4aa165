// noalloc.cu -- np_paged_decode_noalloc: the split decode read (read +
// log-sum-exp merge) for callers that cannot allocate device memory.  The
// split partials live in a fixed array compiled into this library instead of
// a caller-supplied workspace.
#include <atomic>

#include <cuda_runtime.h>

#include "np_paged.h"

namespace {

// Scratch for the split partials.  Every GPU on which the library's kernels
// are loaded holds these NP_NOALLOC_SCRATCH_BYTES bytes until the process
// exits.  Calls never need it zeroed: the read writes every (row, head,
// split) lse and every partial output the merge reads.
static __device__ __align__(256) unsigned char g_noalloc_scratch[NP_NOALLOC_SCRATCH_BYTES];

// Device address of g_noalloc_scratch per device.  In host code the array's
// name only stands for the symbol, so the address comes from
// cudaGetSymbolAddress, once per device, with that device current.
std::atomic<void*> g_scratch_addr[64];

np_status scratch_address(void** addr) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return NP_ERR_CUDA;
  void* p = dev < 64 ? g_scratch_addr[dev].load(std::memory_order_acquire) : nullptr;
  if (p == nullptr) {
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
      return NP_ERR_CUDA;
    if (dev < 64) g_scratch_addr[dev].store(p, std::memory_order_release);
  }
  *addr = p;
  return NP_OK;
}

}  // namespace

extern "C" np_status np_paged_decode_noalloc(
    void* out, const void* q, const void* k_pool, const void* v_pool, np_dtype dtype,
    int64_t num_blocks, int32_t block_size, int32_t kv_heads, int32_t head_dim,
    const int32_t* block_tables, int32_t max_blocks_per_row, const int32_t* context_lens,
    int32_t rows, int32_t query_len, int32_t q_heads, float scale, int32_t num_splits,
    int32_t* err_word, np_stream_t stream) {
  if (num_splits == 1)  // nothing to merge: no scratch involved
    return np_paged_decode(out, q, k_pool, v_pool, dtype, num_blocks, block_size, kv_heads,
                           head_dim, block_tables, max_blocks_per_row, context_lens, rows,
                           query_len, q_heads, scale, num_splits, nullptr, 0, err_word, stream);
  // The shape checks np_paged_decode makes before it looks at a workspace,
  // with its codes, so that a bad shape is never reported as a scratch
  // size problem (and rows * query_len below cannot overflow).
  if (rows < 0 || query_len <= 0 || q_heads <= 0 || head_dim <= 0 || num_splits < 0 ||
      num_splits > 65535)
    return NP_ERR_INVALID_ARG;
  if (rows > 65535 || query_len > 16) return NP_ERR_UNSUPPORTED;
  if (rows == 0) return NP_OK;
  if (num_splits == 0) {  // the balanced read: its cut-row partials go to the scratch
    const size_t need = np_paged_decode_workspace_bytes(rows, q_heads, head_dim, 0);
    if (need == 0 || need > (size_t)NP_NOALLOC_SCRATCH_BYTES) return NP_ERR_WORKSPACE;
    void* ws = nullptr;
    np_status st = scratch_address(&ws);
    if (st != NP_OK) return st;
    return np_paged_decode(out, q, k_pool, v_pool, dtype, num_blocks, block_size, kv_heads,
                           head_dim, block_tables, max_blocks_per_row, context_lens, rows,
                           query_len, q_heads, scale, 0, ws, NP_NOALLOC_SCRATCH_BYTES, err_word,
                           stream);
  }
  if (out == nullptr || reinterpret_cast<uintptr_t>(out) % 16 != 0) return NP_ERR_INVALID_ARG;
  const int64_t units_rows = (int64_t)rows * query_len;  // <= 65535 * 16: fits int32
  const size_t need =
      np_paged_decode_workspace_bytes((int32_t)units_rows, q_heads, head_dim, num_splits);
  if (need == 0 || need > (size_t)NP_NOALLOC_SCRATCH_BYTES) return NP_ERR_WORKSPACE;
  void* ws = nullptr;
  np_status st = scratch_address(&ws);
  if (st != NP_OK) return st;
  st = np_paged_decode(nullptr, q, k_pool, v_pool, dtype, num_blocks, block_size, kv_heads,
                       head_dim, block_tables, max_blocks_per_row, context_lens, rows,
                       query_len, q_heads, scale, num_splits, ws, NP_NOALLOC_SCRATCH_BYTES,
                       err_word, stream);
  if (st != NP_OK) return st;
  return np_paged_decode_reduce(out, dtype, ws, NP_NOALLOC_SCRATCH_BYTES, (int32_t)units_rows,
                                q_heads, head_dim, num_splits, stream);
}
