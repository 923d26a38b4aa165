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

// One CTA of 4 warps per (row, query head).  L = max_s lse_s; out =
// sum_s e^(lse_s-L) o_s / sum_s e^(lse_s-L) over the splits with finite lse;
// zeros if none.  Warp w takes splits w, w+4, ...; its loads are unrolled
// and unconditional (an empty split's o is masked by a select, never
// multiplied), so many rows are in flight at once.  Lane l owns dims
// {4l + 128k}; head_dim <= 256.
constexpr int kReduceWarps = 4;
constexpr int kReduceUnroll = 4;

template <typename TO>
__global__ void __launch_bounds__(32 * kReduceWarps) lse_reduce_kernel(
    TO* __restrict__ out, const float* __restrict__ ws_o, const float* __restrict__ ws_lse,
    int32_t num_splits, int32_t head_dim) {
  constexpr unsigned FULL = 0xffffffffu;
  __shared__ float part[kReduceWarps][2][128 + 4];
  __shared__ float wpart[kReduceWarps];
  const int64_t u = blockIdx.x;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const float* lse = ws_lse + u * num_splits;
  float big = -INFINITY;
  int last = -1;  // the last split holding tokens
  for (int s = lane; s < num_splits; s += 32) {
    const float ls = lse[s];
    big = fmaxf(big, ls);
    if (ls != -INFINITY) last = s;
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    big = fmaxf(big, __shfl_xor_sync(FULL, big, off));
    last = max(last, __shfl_xor_sync(FULL, last, off));
  }
  const int nsplit = last + 1;  // splits past it are empty: never loaded

  float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
  float wsum = 0.f;
  const bool k0 = 4 * lane < head_dim, k1 = 4 * lane + 128 < head_dim;
  if (big != -INFINITY) {
    const float* ob = ws_o + u * num_splits * (int64_t)head_dim + 4 * lane;
    for (int s0 = warp; s0 < nsplit; s0 += kReduceWarps * kReduceUnroll) {
      float w[kReduceUnroll];
      float4 v0[kReduceUnroll], v1[kReduceUnroll];
#pragma unroll
      for (int i = 0; i < kReduceUnroll; ++i) {
        const int s = s0 + i * kReduceWarps;
        const bool in = s < nsplit;
        const float ls = in ? lse[s] : -INFINITY;
        w[i] = (ls == -INFINITY) ? 0.f : expf(ls - big);
        const float* o = ob + (int64_t)(in ? s : 0) * head_dim;
        v0[i] = k0 ? *reinterpret_cast<const float4*>(o) : make_float4(0.f, 0.f, 0.f, 0.f);
        v1[i] = k1 ? *reinterpret_cast<const float4*>(o + 128) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int i = 0; i < kReduceUnroll; ++i) {
        const bool use = w[i] > 0.f;
        wsum += w[i];
        acc[0][0] += use ? w[i] * v0[i].x : 0.f;
        acc[0][1] += use ? w[i] * v0[i].y : 0.f;
        acc[0][2] += use ? w[i] * v0[i].z : 0.f;
        acc[0][3] += use ? w[i] * v0[i].w : 0.f;
        acc[1][0] += use ? w[i] * v1[i].x : 0.f;
        acc[1][1] += use ? w[i] * v1[i].y : 0.f;
        acc[1][2] += use ? w[i] * v1[i].z : 0.f;
        acc[1][3] += use ? w[i] * v1[i].w : 0.f;
      }
    }
  }
#pragma unroll
  for (int k = 0; k < 2; ++k)
#pragma unroll
    for (int e = 0; e < 4; ++e) part[warp][k][4 * lane + e] = acc[k][e];
  if (lane == 0) wpart[warp] = wsum;
  __syncthreads();
  if (warp != 0) return;
  float tot = 0.f;
#pragma unroll
  for (int w2 = 0; w2 < kReduceWarps; ++w2) tot += wpart[w2];
  const float inv = tot > 0.f ? 1.f / tot : 0.f;
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int d = 4 * lane + 128 * k;
    if (d < head_dim) {
      float x[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float a = 0.f;
#pragma unroll
        for (int w2 = 0; w2 < kReduceWarps; ++w2) a += part[w2][k][4 * lane + e];
        x[e] = a * inv;
      }
      Storage<TO>::template store<4>(out + u * head_dim + d, x);
    }
  }
}

np_status launch_reduce(void* out, np_dtype out_dtype, const float* ws_o, const float* ws_lse,
                        int32_t rows, int32_t q_heads, int32_t head_dim, int32_t num_splits,
                        cudaStream_t s) {
  const int64_t units = (int64_t)rows * q_heads;
  if (units == 0) return NP_OK;
  if (units > 0x7fffffffll) return NP_ERR_UNSUPPORTED;
  if (out_dtype == NP_BF16)
    lse_reduce_kernel<__nv_bfloat16><<<(unsigned)units, 32 * kReduceWarps, 0, s>>>(
        static_cast<__nv_bfloat16*>(out), ws_o, ws_lse, num_splits, head_dim);
  else
    lse_reduce_kernel<float><<<(unsigned)units, 32 * kReduceWarps, 0, s>>>(
        static_cast<float*>(out), ws_o, ws_lse, num_splits, head_dim);
  return cudaGetLastError() == cudaSuccess ? NP_OK : NP_ERR_CUDA;
}

// ---------------------------------------------------- bounded-wait check --
// One warp waits, with the pipeline's bounded wait, on an mbarrier that
// nothing will ever complete: after `limit` cycles the wait gives up, the
// kernel flags NP_FLAG_TIMEOUT and returns -- the path every pipeline wait
// takes when its copies never land, exercised without any fault.
__global__ void __launch_bounds__(32) bounded_wait_check_kernel(int32_t* err, long long limit) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);  // expects one arrival; none comes
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncwarp();
  const bool ok = mbar_wait(smem_u32(&bar), 0u, &abort_flag, limit);
  if (!__all_sync(0xffffffffu, ok) && threadIdx.x == 0) set_flag(err, NP_FLAG_TIMEOUT);
}

np_status launch_bounded_wait_check(int32_t* err, long long limit, cudaStream_t stream) {
  bounded_wait_check_kernel<<<1, 32, 0, stream>>>(err, limit);
  return cudaGetLastError() == cudaSuccess ? NP_OK : NP_ERR_CUDA;
}

}  // namespace npk
