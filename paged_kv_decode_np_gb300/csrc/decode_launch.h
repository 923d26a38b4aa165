// decode_launch.h -- host-side interface between the C ABI (api.cu) and the
// per-(dtype, head_dim) decode instantiations (decode_inst.cu).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "np_paged.h"

namespace npk {

struct DecodeParams;

struct DecodeLaunch {
  // filled by the caller
  const DecodeParams* params;  // stages is filled in by the launcher
  int group;                   // G = q_heads / kv_heads
  int head_group;              // HG
  int token_warps;             // TW
  int rows, splits, head_groups;
  bool streamed;               // balanced streamed read: grid = `splits` CTAs
  size_t smem_budget;          // bytes of dynamic shared memory available
  cudaStream_t stream;
  // filled by the launcher
  int stages;
  size_t smem_bytes;
};

// Returns NP_OK, NP_ERR_UNSUPPORTED (group not compiled / ring does not fit)
// or NP_ERR_CUDA.
typedef np_status (*DecodeLauncher)(DecodeLaunch& L, DecodeParams& p);

np_status decode_f32_d16(DecodeLaunch&, DecodeParams&);
np_status decode_f32_d32(DecodeLaunch&, DecodeParams&);
np_status decode_f32_d64(DecodeLaunch&, DecodeParams&);
np_status decode_f32_d128(DecodeLaunch&, DecodeParams&);
np_status decode_f32_d256(DecodeLaunch&, DecodeParams&);
np_status decode_bf16_d16(DecodeLaunch&, DecodeParams&);
np_status decode_bf16_d32(DecodeLaunch&, DecodeParams&);
np_status decode_bf16_d64(DecodeLaunch&, DecodeParams&);
np_status decode_bf16_d128(DecodeLaunch&, DecodeParams&);
np_status decode_bf16_d256(DecodeLaunch&, DecodeParams&);

// append_reduce.cu
np_status launch_append(void* k_pool, void* v_pool, int64_t num_slots, int64_t row_bytes,
                        const void* k_new, const void* v_new, const int64_t* slot_mapping,
                        int32_t num_tokens, int32_t* err, cudaStream_t s);
np_status launch_bounded_wait_check(int32_t* err, long long limit, cudaStream_t stream);
np_status launch_reduce(void* out, np_dtype out_dtype, const float* ws_o, const float* ws_lse,
                        int32_t rows, int32_t q_heads, int32_t head_dim, int32_t num_splits,
                        cudaStream_t s);

}  // namespace npk
