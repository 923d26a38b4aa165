// append_reduce.cu -- the KV append (slot-mapping scatter) and the split
// log-sum-exp reduce.
#include <math.h>

#include "decode_launch.h"
#include "np_common.cuh"

namespace npk {

// One CTA per new token: copies its K row and V row (kv_heads*head_dim
// elements, a multiple of 16 bytes) to pool slot slot_mapping[token] with
// 16-byte vectors.  Negative slot: padding, skipped.  Slot past the pool:
// skipped and flagged.  ("Day 25: the fused read dispatches to the kernel
// backend", What I learned 1: scatter and gather are exact copies.)
__global__ void __launch_bounds__(128) kv_append_kernel(
    uint4* __restrict__ k_pool, uint4* __restrict__ v_pool, const uint4* __restrict__ k_new,
    const uint4* __restrict__ v_new, const int64_t* __restrict__ slot_mapping,
    int64_t num_slots, int64_t row_vec, int32_t* err) {
  const int64_t tok = blockIdx.x;
  const int64_t s = slot_mapping[tok];
  if (s < 0) return;
  if (s >= num_slots) {
    if (threadIdx.x == 0) set_flag(err, NP_FLAG_SLOT);
    return;
  }
  uint4* kd = k_pool + s * row_vec;
  uint4* vd = v_pool + s * row_vec;
  const uint4* ks = k_new + tok * row_vec;
  const uint4* vs = v_new + tok * row_vec;
  for (int64_t i = threadIdx.x; i < row_vec; i += blockDim.x) {
    kd[i] = ks[i];
    vd[i] = vs[i];
  }
}

np_status launch_append(void* k_pool, void* v_pool, int64_t num_slots, int64_t row_bytes,
                        const void* k_new, const void* v_new, const int64_t* slot_mapping,
                        int32_t num_tokens, int32_t* err, cudaStream_t s) {
  if (num_tokens == 0) return NP_OK;
  kv_append_kernel<<<num_tokens, 128, 0, s>>>(
      static_cast<uint4*>(k_pool), static_cast<uint4*>(v_pool),
      static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new), slot_mapping,
      num_slots, row_bytes / 16, err);
  return cudaGetLastError() == cudaSuccess ? NP_OK : NP_ERR_CUDA;
}

// One warp per (row, query head).  L = max_s lse_s; out = sum_s e^(lse_s-L)
// o_s / sum_s e^(lse_s-L) over the splits with finite lse; zeros if none.
// Lane l owns dims {4l + 128k}; head_dim <= 256.
template <typename TO>
__global__ void __launch_bounds__(128) lse_reduce_kernel(TO* __restrict__ out,
                                                         const float* __restrict__ ws_o,
                                                         const float* __restrict__ ws_lse,
                                                         int64_t units, int32_t num_splits,
                                                         int32_t head_dim) {
  constexpr unsigned FULL = 0xffffffffu;
  const int64_t u = (int64_t)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (u >= units) return;
  const float* lse = ws_lse + u * num_splits;
  float big = -INFINITY;
  for (int s = lane; s < num_splits; s += 32) big = fmaxf(big, lse[s]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) big = fmaxf(big, __shfl_xor_sync(FULL, big, off));

  float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
  float wsum = 0.f;
  if (big != -INFINITY) {
    for (int s = 0; s < num_splits; ++s) {
      const float ls = lse[s];
      if (ls == -INFINITY) continue;
      const float w = expf(ls - big);
      wsum += w;
      const float* o = ws_o + (u * num_splits + s) * head_dim;
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int d = 4 * lane + 128 * k;
        if (d < head_dim) {
          const float4 v = *reinterpret_cast<const float4*>(o + d);
          acc[k][0] = fmaf(w, v.x, acc[k][0]);
          acc[k][1] = fmaf(w, v.y, acc[k][1]);
          acc[k][2] = fmaf(w, v.z, acc[k][2]);
          acc[k][3] = fmaf(w, v.w, acc[k][3]);
        }
      }
    }
  }
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int d = 4 * lane + 128 * k;
    if (d < head_dim) {
      float x[4] = {acc[k][0] * inv, acc[k][1] * inv, acc[k][2] * inv, acc[k][3] * inv};
      Storage<TO>::template store<4>(out + u * head_dim + d, x);
    }
  }
}

np_status launch_reduce(void* out, np_dtype out_dtype, const float* ws_o, const float* ws_lse,
                        int32_t rows, int32_t q_heads, int32_t head_dim, int32_t num_splits,
                        cudaStream_t s) {
  const int64_t units = (int64_t)rows * q_heads;
  if (units == 0) return NP_OK;
  const int64_t blocks = (units + 3) / 4;
  if (out_dtype == NP_BF16)
    lse_reduce_kernel<__nv_bfloat16><<<(unsigned)blocks, 128, 0, s>>>(
        static_cast<__nv_bfloat16*>(out), ws_o, ws_lse, units, num_splits, head_dim);
  else
    lse_reduce_kernel<float><<<(unsigned)blocks, 128, 0, s>>>(static_cast<float*>(out), ws_o,
                                                              ws_lse, units, num_splits, head_dim);
  return cudaGetLastError() == cudaSuccess ? NP_OK : NP_ERR_CUDA;
}

}  // namespace npk
