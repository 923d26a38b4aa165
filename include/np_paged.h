/*
 * np_paged.h -- C ABI of the GB300 (sm_103a) batched paged-attention decode
 * library, libnp_paged.so.
 *
 * The operation (one decode step of an inference engine's paged KV cache):
 *
 *   1. np_kv_append: each new token's K and V rows are written into a shared
 *      pool of fixed-size blocks at the flat slot given by a slot mapping,
 *      slot = physical_block * block_size + offset ("Day 25: the fused read
 *      dispatches to the kernel backend", What I added today: the read gets
 *      the layer's K/V pools and a slot mapping covering every history token;
 *      What I learned 1: scatter and gather are exact copies).
 *
 *   2. np_paged_decode: each row's single query token attends over that
 *      row's whole history, which is scattered over the pool and addressed
 *      through the row's block table ("Day 17: paging under the sampling
 *      path", Post angle and Diagram: the cache is a pool of fixed-size
 *      blocks, and each row's block table maps its positions to blocks).  The result equals scaled-dot-product
 *      attention over the gathered history ("Day 25", What I added today),
 *      computed as a streamed (online) softmax that never materialises the
 *      [rows, heads, 1, ctx] array of scores ("Day 60: the read becomes a
 *      choice", What I added today and Post angle).  Query heads share kv
 *      heads in groups (GQA): q head h reads kv head h / (q_heads/kv_heads).
 *
 *   3. np_paged_decode_reduce: when the read is split along the context
 *      (flash-decoding: each split of a row's history is read by its own
 *      thread block), the per-split partial outputs are merged by their
 *      log-sum-exp.  The pages do not describe this split; it is how this
 *      library spreads long and ragged histories over the GPU.
 *
 * Conventions shared by every call:
 *   - Every data pointer is CALLER-OWNED DEVICE memory on the current CUDA
 *     device, dense and row-major in the layout stated for it, 16-byte
 *     aligned.  The library never allocates, frees, or synchronises; it never
 *     reads device memory back to the host, so a step can be captured in a
 *     CUDA graph (after the first call on a device, which sets kernel
 *     attributes).
 *   - Work is enqueued on `stream` (NULL = the legacy default stream) and
 *     runs asynchronously; the return value covers argument validation and
 *     the launch only.  Validation failures return before anything is
 *     enqueued.
 *   - Host threads may call the library concurrently (its only shared state
 *     is per-device launch configuration, set once, and per-thread caches
 *     of tensor maps).  On the device, a workspace belongs to one call in
 *     flight: calls that may overlap (other streams, or a graph replayed
 *     alongside) each need their own workspace, output and err_word.
 *   - Device-side problems never trap or fault: the affected token/block is
 *     skipped or clamped and a bit is OR-ed into *err_word (a device int32
 *     the caller zeroes and reads when convenient; NULL = not reported).
 *   - Pools: k_pool and v_pool are separate arrays, each
 *     [num_blocks, block_size, kv_heads, head_dim] of `dtype`.
 *   - Supported: dtype NP_F32 or NP_BF16; head_dim in {16, 32, 64, 128, 256};
 *     group g = q_heads/kv_heads from 1 to 8 on fp32 pools, from 1 to 16 on
 *     bf16 pools; any block_size >= 1; any kv_heads >= 1; query_len 1, or
 *     any query_len with g * query_len <= 16 on bf16 pools, <= 8 on fp32
 *     pools, on every schedule.  Arithmetic is fp32 in every case (bf16 is
 *     widened exactly); q and out have the pool dtype.
 *   - Several query tokens per row (query_len Q > 1, speculative or chunked
 *     decode): the row's Q query tokens are its last Q positions
 *     c - Q .. c - 1 (c = context_lens[r], counting them); query token i
 *     attends causally to positions 0 .. c - Q + i.  q and out are then
 *     [rows, Q, q_heads, head_dim]; everything sized "per row and head"
 *     below is per (row, query token) and head.
 */
#ifndef NP_PAGED_H
#define NP_PAGED_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define NP_ABI_VERSION 2

/* Same type as cudaStream_t / CUstream, without pulling in CUDA headers. */
typedef struct CUstream_st* np_stream_t;

typedef enum np_status {
  NP_OK = 0,
  NP_ERR_INVALID_ARG = 1,  /* null/misaligned pointer, bad shape or value */
  NP_ERR_UNSUPPORTED = 2,  /* head_dim, group or dtype outside the set above */
  NP_ERR_WORKSPACE = 3,    /* workspace missing or smaller than required */
  NP_ERR_OUT_OF_RANGE = 4, /* a size whose byte count overflows int64 */
  NP_ERR_CUDA = 5          /* a CUDA runtime call or launch failed */
} np_status;

typedef enum np_dtype { NP_F32 = 0, NP_BF16 = 1 } np_dtype;

/* Bits OR-ed into *err_word by the kernels. */
#define NP_FLAG_BLOCK_ID 0x1 /* a block-table entry the walk needed was outside
                                [0, num_blocks); block 0 was read instead */
#define NP_FLAG_CONTEXT 0x2  /* context_lens[r] < 0 or > max_blocks_per_row *
                                block_size; clamped into that range */
#define NP_FLAG_SLOT 0x4     /* an append slot >= num_blocks * block_size, or
                                (np_paged_append_decode) not the slot of the
                                row's newest position; that token was not
                                written */
#define NP_FLAG_TIMEOUT 0x8  /* an internal pipeline wait gave up (never
                                expected; the output of that block is wrong) */
#define NP_FLAG_CONFIG 0x10  /* a thread block found its launch configuration
                                inconsistent and did nothing (never expected) */

/* Human-readable name of a status code (static string, never NULL). */
const char* np_status_string(np_status status);

/* NP_ABI_VERSION of the loaded library. */
int32_t np_abi_version(void);

/*
 * np_kv_append -- scatter this step's new K/V into the pools.
 *   k_pool, v_pool  [num_blocks, block_size, kv_heads, head_dim] dtype (written)
 *   k_new, v_new    [num_tokens, kv_heads, head_dim] dtype
 *   slot_mapping    [num_tokens] int64: token i goes to pool slot
 *                   slot_mapping[i] (element offset slot*kv_heads*head_dim);
 *                   a negative slot means "padding, skip"; a slot
 *                   >= num_blocks*block_size is skipped and flagged
 *                   (NP_FLAG_SLOT).
 * Bit-exact copy.  Two tokens with the same slot: one of them wins
 * (unspecified which).  num_tokens == 0 is a no-op.
 */
np_status np_kv_append(void* k_pool, void* v_pool, np_dtype dtype,
                       int64_t num_blocks, int32_t block_size,
                       int32_t kv_heads, int32_t head_dim, const void* k_new,
                       const void* v_new, const int64_t* slot_mapping,
                       int32_t num_tokens, int32_t* err_word,
                       np_stream_t stream);

/*
 * np_paged_decode_plan -- the schedule the library recommends, as a
 * num_splits value for np_paged_decode.  Pure host arithmetic on STATIC
 * shapes only (never on context_lens, so the choice needs no device read and
 * a step stays graph-capturable).  num_sms <= 0 queries the current device's
 * SM count.  Writes 0 (the balanced read) when the shapes allow it, else a
 * split count >= 1 sized to about 2 MB of K+V per thread block.
 */
np_status np_paged_decode_plan(int32_t rows, int32_t q_heads, int32_t kv_heads,
                               int32_t head_dim, int32_t block_size,
                               int32_t max_blocks_per_row, np_dtype dtype,
                               int32_t num_sms, int32_t* num_splits);

/*
 * np_paged_decode_split_len -- tokens per split for a given split count:
 * ceil(max_blocks_per_row*block_size / num_splits) rounded up to a multiple
 * of 64 tokens (and of block_size when block_size > 64).  Split s covers
 * history tokens [s*split_len, (s+1)*split_len).  Returns -1 on bad input.
 */
int64_t np_paged_decode_split_len(int32_t block_size,
                                  int32_t max_blocks_per_row,
                                  int32_t num_splits);

/*
 * np_paged_decode_workspace_bytes -- workspace a read needs:
 *   num_splits > 1: partial outputs [rows, q_heads, num_splits, head_dim]
 *                   fp32 at offset 0, partial lse [rows, q_heads,
 *                   num_splits] fp32 at the next 256-byte boundary (natural
 *                   log; -inf for an empty split).  For query_len > 1 pass
 *                   rows * query_len as `rows`.
 *   num_splits == 0 (balanced read): a fixed size that depends on head_dim
 *                   only (partials of the rows cut between thread blocks);
 *                   its layout is private to the library.
 *   0 when num_splits == 1.  No read needs the workspace initialised.
 */
size_t np_paged_decode_workspace_bytes(int32_t rows, int32_t q_heads,
                                       int32_t head_dim, int32_t num_splits);

/*
 * np_paged_decode -- the decode read.
 *   out            [rows, query_len, q_heads, head_dim] dtype; written when
 *                  num_splits == 1 (may be NULL otherwise)
 *   q              [rows, query_len, q_heads, head_dim] dtype
 *   query_len      query tokens per row (1 = the usual decode step)
 *   k_pool, v_pool [num_blocks, block_size, kv_heads, head_dim] dtype
 *   block_tables   [rows, max_blocks_per_row] int32: logical block j of row
 *                  r is physical block block_tables[r*max_blocks_per_row+j];
 *                  entries at j >= ceil(context_lens[r]/block_size) are
 *                  never read
 *   context_lens   [rows] int32: history length of each row (including any
 *                  token appended this step); 0 gives an all-zero output
 *   scale          softmax scale applied to q.k (finite)
 *   num_splits     >= 0.  1: out is written directly.  > 1: split s of row r
 *                  (tokens [s*split_len, (s+1)*split_len), see
 *                  np_paged_decode_split_len) writes its normalised partial
 *                  output and lse into `workspace`; call
 *                  np_paged_decode_reduce next to produce out.
 *                  0: the balanced read -- one thread block per SM (at most
 *                  160), each taking an equal share (in chunks) of all
 *                  rows' history laid end to end (computed on the device
 *                  from context_lens); rows cut between blocks are merged
 *                  by a second launch on `stream`, each cut row's merge
 *                  spread over the blocks that read it, in block order
 *                  (results are deterministic).  out is written; no reduce
 *                  call.
 *                  Needs head_dim a multiple of 64 (bf16) or 32 (fp32, up
 *                  to 256); any kv_heads, taken HG at a time (HG = the
 *                  largest divisor of kv_heads up to 8); for bf16,
 *                  box_tokens * HG a multiple of 8, where box_tokens is the
 *                  largest power of two dividing block_size, at most 16 (8
 *                  at head_dim 256) -- e.g. block_size a multiple of 8 when
 *                  HG = 1; rows * kv_heads / HG <= 4096, tables of at most
 *                  2^31 - 1 tokens and a workspace (else NP_ERR_UNSUPPORTED
 *                  / NP_ERR_WORKSPACE).
 *                  Results equal the split read's up to fp32 rounding order.
 *   workspace      device buffer of >= np_paged_decode_workspace_bytes(...)
 *                  bytes, 256-byte aligned (may be NULL when num_splits == 1)
 *   err_word       device int32 or NULL (NP_FLAG_BLOCK_ID, NP_FLAG_CONTEXT,
 *                  NP_FLAG_TIMEOUT)
 * Memory traffic: each history token's K and V rows are read once from HBM;
 * q, block tables and context lengths once; out (or the partials) written
 * once.
 */
np_status np_paged_decode(void* out, const void* q, const void* k_pool,
                          const void* v_pool, np_dtype dtype,
                          int64_t num_blocks, int32_t block_size,
                          int32_t kv_heads, int32_t head_dim,
                          const int32_t* block_tables,
                          int32_t max_blocks_per_row,
                          const int32_t* context_lens, int32_t rows,
                          int32_t query_len, int32_t q_heads, float scale,
                          int32_t num_splits, void* workspace,
                          size_t workspace_bytes, int32_t* err_word,
                          np_stream_t stream);

/*
 * np_paged_append_decode -- np_kv_append of the rows' new tokens followed
 * by np_paged_decode, in ONE kernel launch (same results, bit for bit in
 * the pools).  Row r's query_len new tokens (k_new/v_new [rows, query_len,
 * kv_heads, head_dim]) go to pool slots slot_mapping[r*query_len + j]
 * ([rows, query_len] int64), which must be the slots of the row's newest
 * positions, context_lens[r] - query_len + j, under its block table (the
 * usual decode step: append, then read the whole history); a negative entry
 * means "no new token here".  The thread block whose split holds a position
 * writes that token before it reads it.  An entry that names any other slot
 * is not written and is flagged (NP_FLAG_SLOT) -- use np_kv_append +
 * np_paged_decode for arbitrary slots.  Other arguments, layouts and errors
 * as np_paged_decode; with num_splits > 1, call np_paged_decode_reduce next.
 */
np_status np_paged_append_decode(void* out, const void* q, const void* k_new,
                                 const void* v_new, const int64_t* slot_mapping,
                                 void* k_pool, void* v_pool, np_dtype dtype,
                                 int64_t num_blocks, int32_t block_size,
                                 int32_t kv_heads, int32_t head_dim,
                                 const int32_t* block_tables,
                                 int32_t max_blocks_per_row,
                                 const int32_t* context_lens, int32_t rows,
                                 int32_t query_len, int32_t q_heads,
                                 float scale, int32_t num_splits,
                                 void* workspace, size_t workspace_bytes,
                                 int32_t* err_word, np_stream_t stream);

/*
 * np_paged_decode_reduce -- merge split partials into out.
 *   out        [rows, q_heads, head_dim] of out_dtype (for query_len > 1:
 *              pass rows * query_len as `rows`)
 *   workspace  as written by np_paged_decode with the same rows, q_heads,
 *              head_dim and num_splits
 * For each (row, head): L = max_s lse_s; out = sum_s e^(lse_s - L) o_s /
 * sum_s e^(lse_s - L), skipping splits whose lse is -inf; all splits empty
 * gives zeros.
 */
np_status np_paged_decode_reduce(void* out, np_dtype out_dtype,
                                 const void* workspace, size_t workspace_bytes,
                                 int32_t rows, int32_t q_heads,
                                 int32_t head_dim, int32_t num_splits,
                                 np_stream_t stream);

/*
 * np_paged_decode_noalloc -- np_paged_decode followed by
 * np_paged_decode_reduce, for callers that cannot allocate device memory.
 * The pages have no counterpart to this call; it exists for callers that
 * are handed their inputs, outputs and a stream and nothing else -- a host
 * framework calling this library as a plugin without exposing its
 * allocator, or a serving loop that must not allocate once it is running
 * (cudaMalloc can synchronise the device and can fail under memory
 * pressure).  Such callers cannot provide the split workspace, so this
 * call keeps the split partials in a fixed array compiled into the library:
 * NP_NOALLOC_SCRATCH_BYTES of device memory that every GPU loading the
 * library holds until the process exits.
 *
 * Arguments, layouts and errors are those of np_paged_decode, with `out`
 * always written and no workspace.  It allocates and frees nothing.
 *   - Returns NP_ERR_WORKSPACE, before anything is enqueued, when the
 *     partials, np_paged_decode_workspace_bytes(rows * query_len, q_heads,
 *     head_dim, num_splits), exceed NP_NOALLOC_SCRATCH_BYTES; a smaller
 *     num_splits fits.  num_splits == 1 uses no scratch at all;
 *     num_splits == 0 (the balanced read) keeps its cut-row partials there
 *     (it fits for head_dim <= 128).
 *   - The first call on a device looks up the array's device address for
 *     that device (cudaGetSymbolAddress) and keeps it for the life of the
 *     process; make that first call before any stream capture.  Tearing the
 *     device's context down (cudaDeviceReset) can move the array, and the
 *     kept address then points at nothing: do not call this entry point on
 *     a device after resetting it.
 *   - Sizes np_paged_decode refuses (negative rows; query_len, q_heads or
 *     head_dim below 1; num_splits outside 0..65535: NP_ERR_INVALID_ARG; rows above
 *     65535 or query_len above 16: NP_ERR_UNSUPPORTED) are refused with the
 *     same codes before the scratch size is compared.
 *   - Every call on a device shares the one array, which keeps the last
 *     call's contents (nothing in it needs to start zeroed).  Calls whose
 *     execution overlaps on the GPU (different streams, or overlapping
 *     graph launches) race on it: order them on one stream.
 */
#define NP_NOALLOC_SCRATCH_BYTES (32u << 20) /* 32 MiB per device */

np_status np_paged_decode_noalloc(void* out, const void* q, const void* k_pool,
                                  const void* v_pool, np_dtype dtype,
                                  int64_t num_blocks, int32_t block_size,
                                  int32_t kv_heads, int32_t head_dim,
                                  const int32_t* block_tables,
                                  int32_t max_blocks_per_row,
                                  const int32_t* context_lens, int32_t rows,
                                  int32_t query_len, int32_t q_heads,
                                  float scale, int32_t num_splits,
                                  int32_t* err_word, np_stream_t stream);

/*
 * np_selftest_bounded_wait -- checks, on the device, the failure path every
 * pipeline wait of the read takes when its copies never land: one warp waits
 * on an mbarrier that nothing completes, gives up after limit_cycles SM
 * clock cycles (1 .. 2e9; 2e9 is the read's own limit, about 1 s), ORs
 * NP_FLAG_TIMEOUT into *err_word (device int32, required) and returns; the
 * context stays usable.  Nothing faults or traps.  For health checks and
 * tests; not part of a decode step.
 */
np_status np_selftest_bounded_wait(int32_t* err_word, int64_t limit_cycles,
                                   np_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* NP_PAGED_H */
